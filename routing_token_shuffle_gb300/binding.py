"""Thin ctypes binding of libsmoe.so (include/smoe.h).

Argument marshalling only: every function here forwards device pointers of torch
tensors (or raw integers) to the C entry point of the same name and raises
``SmoeError`` on a non-zero status. No step of the layer runs in Python. If the
library has not been built, loading it raises immediately; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libsmoe.so")

SMOE_F32, SMOE_BF16 = 0, 1

STATUS = {
    0: "SMOE_OK", -1: "SMOE_ERR_ARG", -2: "SMOE_ERR_SHAPE", -3: "SMOE_ERR_ALIGN",
    -4: "SMOE_ERR_WORKSPACE", -5: "SMOE_ERR_CUDA", -6: "SMOE_ERR_DATA",
    -7: "SMOE_ERR_DEVICE_TIMEOUT", -8: "SMOE_ERR_UNSUPPORTED",
}


class SmoeError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__(f"{fn} -> {STATUS.get(code, code)}: {msg}")
        self.code = code


class SmoeDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "E", "K", "H", "F", "n_shared", "P", "vocab", "dtype", "renorm")]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_gate", "w1", "w3", "w2", "conf", "expert_part")]


class LayerIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("x", "token_ids", "y", "logits", "topk_idx", "topk_w", "pred_part", "shuf_perm",
                 "part_off", "expert_off", "pair_row", "row_token", "lar")] + [
                   ("skip_shuffle", ctypes.c_int32)]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_D = ctypes.POINTER(SmoeDesc)

SIGNATURES = {
    "smoe_workspace_size": (_SZ, [_D]),
    "smoe_route": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_predict_shuffle": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_predict_shuffle_noalloc": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "smoe_lar": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_token_cluster": (ctypes.c_int, [_D, _P, _P, _P, _P, _SZ, _P]),
    "smoe_predict_shuffle_inter": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                  _SZ, _P]),
    "smoe_dispatch": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_shuffle_dispatch_rows": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_expert_ffn": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_expert_ffn_gather": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                              _SZ, _P]),
    "smoe_expert_ffn_gather_fused": (ctypes.c_int, [_D]),
    "smoe_combine": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_ep_exchange": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_srs": (ctypes.c_int, [_D, ctypes.c_int, _P, _P, _P, _P, _SZ, _P]),
    "smoe_sag": (ctypes.c_int, [_D, _P, _P, _P, _P, _SZ, _P]),
    "smoe_layer_forward": (ctypes.c_int, [_D, ctypes.POINTER(LayerWeights),
                                          ctypes.POINTER(LayerIO), _P, _SZ, _P]),
    "smoe_layer_forward_host": (ctypes.c_int, [_D, ctypes.POINTER(LayerWeights), _P, _P, _P, _P,
                                               _SZ, _P]),
    "smoe_prefetch_predict": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             _P, _SZ, _P]),
    "smoe_moe_forward_routed": (ctypes.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "smoe_get_status": (ctypes.c_int, [_P, _P]),
    "smoe_selftest_device_timeout": (ctypes.c_int, [_P, _SZ, _P]),
    "smoe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "smoe_last_error": (ctypes.c_char_p, []),
    "smoe_kernel_launches": (ctypes.c_ulonglong, []),
}

_lib = None


def lib(path: str | None = None):
    """Load libsmoe.so once (from ``path``, else LIB_PATH); raise if it is missing (no
    fallback path exists)."""
    global _lib
    if _lib is None:
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run routing_token_shuffle_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    """A tensor's address, or a raw integer address passed through. Every buffer of the C
    ABI is dense row-major, so a strided view (a transpose, a column slice, an expand)
    is refused here instead of being read as if it were dense."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {t.stride()} is not "
                         "contiguous; the C ABI takes dense row-major buffers (call .contiguous())")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, fn: str):
    if rc != 0:
        raise SmoeError(rc, fn, lib().smoe_last_error().decode())


def make_desc(T, d, E, K, H, F, n_shared, P, vocab, dtype, renorm=0) -> SmoeDesc:
    dt = SMOE_F32 if dtype in ("f32", SMOE_F32) else SMOE_BF16
    return SmoeDesc(T, d, E, K, H, F, n_shared, P, vocab, dt, renorm)


def desc_from_config(cfg, T=None) -> SmoeDesc:
    return make_desc(cfg.T if T is None else T, cfg.d, cfg.E, cfg.K, cfg.H, cfg.F, cfg.n_shared,
                     cfg.P, cfg.vocab, cfg.dtype)


def workspace_size(desc: SmoeDesc) -> int:
    return lib().smoe_workspace_size(ctypes.byref(desc))


def workspace(desc: SmoeDesc, device="cuda"):
    """A zeroed workspace tensor (the status word must start at zero)."""
    import torch
    n = workspace_size(desc)
    if n == 0:
        raise SmoeError(-2, "smoe_workspace_size", "invalid descriptor")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def smoe_route(desc, x, w_gate, topk_idx, topk_w, logits_in=None, logits_out=None, ws=None,
               stream=None):
    nbytes = ws.numel() if ws is not None else 0
    _check(lib().smoe_route(ctypes.byref(desc), _ptr(x), _ptr(w_gate), _ptr(logits_in),
                            _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), nbytes,
                            _stream(stream)), "smoe_route")


def smoe_predict_shuffle(desc, token_ids, conf, expert_part, pred_part, shuf_perm, part_off, ws,
                         x=None, x_shuf=None, stream=None):
    _check(lib().smoe_predict_shuffle(ctypes.byref(desc), _ptr(token_ids), _ptr(conf),
                                      _ptr(expert_part), _ptr(x), _ptr(pred_part), _ptr(shuf_perm),
                                      _ptr(part_off), _ptr(x_shuf), _ptr(ws), ws.numel(),
                                      _stream(stream)), "smoe_predict_shuffle")


def smoe_predict_shuffle_noalloc(desc, token_ids, conf, expert_part, pred_part, shuf_perm,
                                 part_off, x=None, x_shuf=None, stream=None):
    """smoe_predict_shuffle without a workspace (library-held scratch; see smoe.h)."""
    _check(lib().smoe_predict_shuffle_noalloc(ctypes.byref(desc), _ptr(token_ids), _ptr(conf),
                                              _ptr(expert_part), _ptr(x), _ptr(pred_part),
                                              _ptr(shuf_perm), _ptr(part_off), _ptr(x_shuf),
                                              _stream(stream)), "smoe_predict_shuffle_noalloc")


def smoe_token_cluster(desc, topk_idx, expert_part, cluster, ws, stream=None):
    _check(lib().smoe_token_cluster(ctypes.byref(desc), _ptr(topk_idx), _ptr(expert_part),
                                    _ptr(cluster), _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_token_cluster")


def smoe_predict_shuffle_inter(desc, token_ids, conf, expert_part, prev_cluster, table_a,
                               pred_part, shuf_perm, part_off, ws, x=None, x_shuf=None,
                               stream=None):
    _check(lib().smoe_predict_shuffle_inter(
        ctypes.byref(desc), _ptr(token_ids), _ptr(conf), _ptr(expert_part), _ptr(prev_cluster),
        _ptr(table_a), _ptr(x), _ptr(pred_part), _ptr(shuf_perm), _ptr(part_off), _ptr(x_shuf),
        _ptr(ws), ws.numel(), _stream(stream)), "smoe_predict_shuffle_inter")


def smoe_lar(desc, topk_idx, expert_part, counts, ws, src_part=None, stream=None):
    _check(lib().smoe_lar(ctypes.byref(desc), _ptr(topk_idx), _ptr(src_part), _ptr(expert_part),
                          _ptr(counts), _ptr(ws), ws.numel(), _stream(stream)), "smoe_lar")


def smoe_dispatch(desc, topk_idx, expert_off, pair_row, row_token, ws, shuf_perm=None, x_src=None,
                  x_disp=None, row_slot=None, stream=None):
    _check(lib().smoe_dispatch(ctypes.byref(desc), _ptr(topk_idx), _ptr(shuf_perm), _ptr(x_src),
                               _ptr(expert_off), _ptr(pair_row), _ptr(row_token), _ptr(row_slot),
                               _ptr(x_disp), _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_dispatch")


def smoe_shuffle_dispatch_rows(desc, x, pair_row, x_disp, ws, shuf_perm=None, x_shuf=None,
                               stream=None):
    _check(lib().smoe_shuffle_dispatch_rows(ctypes.byref(desc), _ptr(x), _ptr(shuf_perm),
                                            _ptr(pair_row), _ptr(x_shuf), _ptr(x_disp), _ptr(ws),
                                            ws.numel(), _stream(stream)),
           "smoe_shuffle_dispatch_rows")


def smoe_expert_ffn(desc, x_disp, expert_off, w1, w3, w2, y_disp, ws, x=None, y_shared=None,
                    stream=None):
    _check(lib().smoe_expert_ffn(ctypes.byref(desc), _ptr(x_disp), _ptr(x), _ptr(expert_off),
                                 _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y_disp), _ptr(y_shared),
                                 _ptr(ws), ws.numel(), _stream(stream)), "smoe_expert_ffn")


def smoe_expert_ffn_gather(desc, x_src, row_slot, x_disp, expert_off, w1, w3, w2, y_disp, ws,
                           x=None, y_shared=None, stream=None):
    _check(lib().smoe_expert_ffn_gather(ctypes.byref(desc), _ptr(x_src), _ptr(row_slot), _ptr(x),
                                        _ptr(x_disp), _ptr(expert_off), _ptr(w1), _ptr(w3),
                                        _ptr(w2), _ptr(y_disp), _ptr(y_shared), _ptr(ws),
                                        ws.numel(), _stream(stream)), "smoe_expert_ffn_gather")


def smoe_expert_ffn_gather_fused(desc) -> bool:
    return bool(lib().smoe_expert_ffn_gather_fused(ctypes.byref(desc)))


def smoe_combine(desc, y_disp, pair_row, topk_w, y_out, ws, y_shared=None, stream=None):
    _check(lib().smoe_combine(ctypes.byref(desc), _ptr(y_disp), _ptr(pair_row), _ptr(topk_w),
                              _ptr(y_shared), _ptr(y_out), _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_combine")


def smoe_ep_exchange(desc, topk_idx, expert_part, send_counts, recv_off, pair_recv, recv_token,
                     ws, src_part=None, x=None, x_recv=None, stream=None):
    _check(lib().smoe_ep_exchange(ctypes.byref(desc), _ptr(topk_idx), _ptr(src_part),
                                  _ptr(expert_part), _ptr(x), _ptr(send_counts), _ptr(recv_off),
                                  _ptr(pair_recv), _ptr(recv_token), _ptr(x_recv), _ptr(ws),
                                  ws.numel(), _stream(stream)), "smoe_ep_exchange")


def smoe_srs(desc, x_parts, shuf_perm, x_shuf, ws, stream=None):
    """x_parts [R, T, d]; R is taken from its leading dimension."""
    _check(lib().smoe_srs(ctypes.byref(desc), int(x_parts.shape[0]), _ptr(x_parts),
                          _ptr(shuf_perm), _ptr(x_shuf), _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_srs")


def smoe_sag(desc, y_shuf, shuf_perm, y, ws, stream=None):
    _check(lib().smoe_sag(ctypes.byref(desc), _ptr(y_shuf), _ptr(shuf_perm), _ptr(y), _ptr(ws),
                          ws.numel(), _stream(stream)), "smoe_sag")


def layer_weights(w_gate, w1, w3, w2, conf, expert_part) -> LayerWeights:
    return LayerWeights(*(_ptr(t) for t in (w_gate, w1, w3, w2, conf, expert_part)))


def layer_io(x, token_ids, y, **outs) -> LayerIO:
    io = LayerIO()
    io.x, io.token_ids, io.y = _ptr(x), _ptr(token_ids), _ptr(y)
    for k, v in outs.items():
        if k == "skip_shuffle":
            io.skip_shuffle = int(v)
        else:
            setattr(io, k, _ptr(v))
    return io


def smoe_layer_forward(desc, weights: LayerWeights, io: LayerIO, ws, stream=None):
    _check(lib().smoe_layer_forward(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(io),
                                    _ptr(ws), ws.numel(), _stream(stream)), "smoe_layer_forward")


def smoe_layer_forward_host(desc, weights: LayerWeights, x_host, ids_host, y_host, ws,
                            stream=None):
    _check(lib().smoe_layer_forward_host(ctypes.byref(desc), ctypes.byref(weights), _ptr(x_host),
                                         _ptr(ids_host), _ptr(y_host), _ptr(ws), ws.numel(),
                                         _stream(stream)), "smoe_layer_forward_host")


def smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, w_gate_next, pred_idx, true_idx, hits, ws,
                          logits_q=None, logits_s=None, qs_out=None, stream=None):
    _check(lib().smoe_prefetch_predict(ctypes.byref(desc), _ptr(r), _ptr(d_l), _ptr(y), _ptr(gamma),
                                       _ptr(beta), _ptr(w_gate_next), _ptr(logits_q),
                                       _ptr(logits_s), _ptr(pred_idx), _ptr(true_idx), _ptr(hits),
                                       _ptr(qs_out), _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_prefetch_predict")


def smoe_moe_forward_routed(desc, x, topk_idx, topk_w, w1, w3, w2, y, ws, stream=None):
    _check(lib().smoe_moe_forward_routed(ctypes.byref(desc), _ptr(x), _ptr(topk_idx),
                                         _ptr(topk_w), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y),
                                         _ptr(ws), ws.numel(), _stream(stream)),
           "smoe_moe_forward_routed")


def kernel_launches() -> int:
    """Kernels launched through the library by this host thread so far."""
    return int(lib().smoe_kernel_launches())


def smoe_get_status(ws, stream=None):
    _check(lib().smoe_get_status(_ptr(ws), _stream(stream)), "smoe_get_status")


def smoe_selftest_device_timeout(ws, stream=None):
    _check(lib().smoe_selftest_device_timeout(_ptr(ws), ws.numel(), _stream(stream)),
           "smoe_selftest_device_timeout")
