"""Python binding of the int4g C ABI (libfl_int4g.so, declared in include/fl_int4g.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  The library
is loaded lazily and a missing library is an error: there is no fallback.

Function names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "lib", "Int4gError", "FL_SOFTMAX", "FL_SIGMOID", "GROUP",
    "fl_strerror", "fl_int4g_version", "fl_int4g_status",
    "fl_int4g_quantize", "fl_int4g_repacked_bytes", "fl_int4g_repack", "fl_int4g_unrepack",
    "fl_int4g_linear_workspace", "fl_int4g_linear", "fl_int4g_linear_noalloc", "fl_int4g_linear_noalloc_status",
    "fl_int4g_linear_g", "fl_moe_int4g_g",
    "fl_int4g_test_withhold_cluster_arrival", "fl_int4g_test_decode_plan",
    "fl_moe_int4g_workspace", "fl_moe_int4g", "fl_moe_int4g_ptrs", "FlMoeRouting", "fl_int4g_mlp_workspace",
    "fl_moe_router_logits_workspace", "fl_moe_router_logits",
    "fl_int4g_mlp", "fl_int4g_mlp_fused",
]

GROUP = 128
FL_SOFTMAX = 0
FL_SIGMOID = 1

_c_size_p = ctypes.POINTER(ctypes.c_size_t)
_vp = ctypes.c_void_p
_i = ctypes.c_int


class FlMoeRouting(ctypes.Structure):
    """struct fl_moe_routing (routing options of fl_moe_int4g_ex)."""
    _fields_ = [("scoring", ctypes.c_int), ("renorm", ctypes.c_int), ("score_bias", ctypes.c_void_p),
                ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int), ("routed_scale", ctypes.c_float)]


# C signatures: name -> (restype, argtypes)
SIGNATURES = {
    "fl_strerror": (ctypes.c_char_p, [_i]),
    "fl_int4g_version": (_i, []),
    "fl_int4g_status": (_i, [_vp, _vp, ctypes.POINTER(_i)]),
    "fl_int4g_quantize": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "fl_int4g_repacked_bytes": (_i, [_i, _i, _i, _c_size_p]),
    "fl_int4g_repack": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, ctypes.c_size_t, _vp]),
    "fl_int4g_unrepack": (_i, [_vp, ctypes.c_size_t, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "fl_int4g_linear_workspace": (_i, [_i, _i, _i, _c_size_p]),
    "fl_int4g_linear": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_int4g_linear_g": (_i, [_vp, _i, _i, _vp, _i, _i, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_moe_int4g_g": (_i, [_vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(FlMoeRouting), _i, _vp, _vp, _vp, _vp,
                            _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_int4g_linear_noalloc": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp]),
    "fl_int4g_linear_noalloc_status": (_i, [_vp, ctypes.POINTER(_i)]),
    "fl_int4g_test_withhold_cluster_arrival": (_i, [ctypes.c_longlong]),
    "fl_int4g_test_decode_plan": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_longlong)]),
    "fl_moe_int4g_workspace": (_i, [_i, _i, _i, _i, _i, _i, _c_size_p]),
    "fl_int4g_mlp_workspace": (_i, [_i, _i, _i, _c_size_p]),
    "fl_moe_router_logits_workspace": (_i, [_i, _i, _i, _c_size_p]),
    "fl_moe_router_logits": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_int4g_mlp": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_int4g_mlp_fused": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_moe_int4g": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                          _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_moe_int4g_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(FlMoeRouting), _vp, _vp, _vp, _vp,
                             _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fl_moe_int4g_ptrs": (_i, [_vp, _vp, _i, _i, _i, _i, _i, ctypes.POINTER(FlMoeRouting), _vp, _vp, _vp, _vp,
                               _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
}

_LIB = None


class Int4gError(RuntimeError):
    def __init__(self, where, code):
        super().__init__(f"{where}: {fl_strerror(code)} (status {code})")
        self.code = code


def lib():
    """The loaded C library (ctypes.CDLL).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
        L = ctypes.CDLL(_build.LIB)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _torch():
    import torch
    return torch


def _check(where, rc):
    if rc != 0:
        raise Int4gError(where, rc)


def _stream(stream=None):
    torch = _torch()
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:   # the current stream's handle without building a Stream object
        return ctypes.c_void_p(raw(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


_WS = {}


def _workspace(nbytes, device):
    """A zero-filled workspace per (device, stream), grown on demand."""
    torch = _torch()
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _WS.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = buf
    return buf


# ------------------------------------------------------------------ wrappers

def fl_strerror(code):
    return lib().fl_strerror(code).decode()


def fl_int4g_version():
    return lib().fl_int4g_version()


def fl_int4g_status(ws, stream=None):
    out = ctypes.c_int(0)
    _check("fl_int4g_status", lib().fl_int4g_status(_p(ws), _stream(stream), ctypes.byref(out)))
    return out.value


def fl_int4g_repacked_bytes(N, K, group=GROUP):
    out = ctypes.c_size_t(0)
    _check("fl_int4g_repacked_bytes", lib().fl_int4g_repacked_bytes(N, K, group, ctypes.byref(out)))
    return out.value


def fl_int4g_quantize(w, group=GROUP, check=True):
    """fp32 [N, K] CUDA tensor -> canonical (q uint8 [N, K/2], scales int16
    [N, G] holding fp16 bits, zeros uint8 [N, ceil(G/2)])."""
    torch = _torch()
    N, K = w.shape
    G = K // group
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, G), dtype=torch.int16, device=w.device)
    z = torch.empty((N, (G + 1) // 2), dtype=torch.uint8, device=w.device)
    st = torch.zeros(4, dtype=torch.int32, device=w.device)
    _check("fl_int4g_quantize", lib().fl_int4g_quantize(_p(w), N, K, group, _p(q), _p(s), _p(z), _p(st), _stream()))
    if check:
        _check("fl_int4g_quantize (device)", fl_int4g_status(st))
    return q, s, z


def fl_int4g_repack(q, s, z, N, K, group=GROUP):
    torch = _torch()
    nbytes = fl_int4g_repacked_bytes(N, K, group)
    w = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check("fl_int4g_repack",
           lib().fl_int4g_repack(_p(q), _p(s), _p(z), N, K, group, _p(w), nbytes, _stream()))
    return w


def fl_int4g_unrepack(w, N, K, group=GROUP):
    torch = _torch()
    G = K // group
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, G), dtype=torch.int16, device=w.device)
    z = torch.empty((N, (G + 1) // 2), dtype=torch.uint8, device=w.device)
    _check("fl_int4g_unrepack",
           lib().fl_int4g_unrepack(_p(w), w.numel(), N, K, group, _p(q), _p(s), _p(z), _stream()))
    return q, s, z


def fl_int4g_linear_workspace(M, N, K):
    out = ctypes.c_size_t(0)
    _check("fl_int4g_linear_workspace", lib().fl_int4g_linear_workspace(M, N, K, ctypes.byref(out)))
    return out.value


def fl_int4g_linear(x, w, N, y=None, ws=None, group=GROUP):
    """y[M, N] bf16 = x[M, K] bf16 . deq(W)^T, W given in the interleaved
    layout of groups of `group` (128 and 256 share one layout; 64 adds the
    side array: fl_int4g_linear_g)."""
    torch = _torch()
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:   # (a caller's workspace is checked for size by the library)
        ws = _workspace(fl_int4g_linear_workspace(M, N, K), x.device)
    if group == GROUP:
        _check("fl_int4g_linear",
               lib().fl_int4g_linear(_p(x), M, K, _p(w), N, _p(y), _p(ws), ws.numel(), _stream()))
    else:
        _check("fl_int4g_linear_g",
               lib().fl_int4g_linear_g(_p(x), M, K, _p(w), N, int(group), _p(y), _p(ws), ws.numel(), _stream()))
    return y


def fl_int4g_linear_noalloc(x, w, N, y=None):
    """Decode linear (M <= 32) with no workspace: for callers that cannot
    allocate device memory where they call.  The library keeps the scratch in
    a fixed device array shared by all calls (do not overlap calls on the GPU);
    make the first call on a device before any stream capture."""
    torch = _torch()
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check("fl_int4g_linear_noalloc", lib().fl_int4g_linear_noalloc(_p(x), M, K, _p(w), N, _p(y), _stream()))
    return y


def fl_int4g_linear_noalloc_status(stream=None):
    """Reads and clears the status block of fl_int4g_linear_noalloc's
    library-held array on the current device (synchronizes the stream)."""
    out = ctypes.c_int(0)
    _check("fl_int4g_linear_noalloc_status", lib().fl_int4g_linear_noalloc_status(_stream(stream), ctypes.byref(out)))
    return out.value


def fl_int4g_test_withhold_cluster_arrival(ns):
    """Test hook: ns >= 0 makes the cluster reductions of later decode
    launches withhold one arrival, so their bounded wait runs out after ns
    nanoseconds and FL_ERR_TIMEOUT is recorded; ns < 0 turns it off."""
    lib().fl_int4g_test_withhold_cluster_arrival(int(ns))


def fl_int4g_test_decode_plan(M, N, K, sms, group=GROUP, glu=False, minb=0, max_cs=8):
    """Test hook: the decode kernel's plan for one shape, computed on the
    host without a GPU.  A dict of T, G, P, csize, stages, stage_bytes, smem,
    xr_stride, xr_off, red_off and zrow_off, or None when the kernel does not
    take the shape."""
    out = (ctypes.c_longlong * 11)()
    rc = lib().fl_int4g_test_decode_plan(M, N, K, sms, group, int(bool(glu)), minb, max_cs, out)
    if rc != 0:
        return None
    keys = ("T", "G", "P", "csize", "stages", "stage_bytes", "smem", "xr_stride", "xr_off", "red_off", "zrow_off")
    return dict(zip(keys, list(out)))


def fl_int4g_mlp_workspace(M, H, I):
    out = ctypes.c_size_t(0)
    _check("fl_int4g_mlp_workspace", lib().fl_int4g_mlp_workspace(M, H, I, ctypes.byref(out)))
    return out.value


def fl_int4g_mlp(x, w_gate, w_up, w_down, I, y=None, ws=None, one_launch=False):
    """Decode MLP block (M <= 8): y = D . (silu(G x) * (U x)), the three
    matrices in the interleaved layout (G, U: [I, H]; D: [H, I]).
    one_launch: the cooperative single-launch form (fl_int4g_mlp_fused)."""
    torch = _torch()
    M, H = x.shape
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    nb = fl_int4g_mlp_workspace(M, H, I)
    if ws is None:
        ws = _workspace(nb, x.device)
    name = "fl_int4g_mlp_fused" if one_launch else "fl_int4g_mlp"
    _check(name, getattr(lib(), name)(_p(x), M, H, I, _p(w_gate), _p(w_up), _p(w_down), _p(y), _p(ws),
                                      ws.numel(), _stream()))
    return y


def fl_moe_int4g_workspace(M, E, k, H, I, has_shared):
    out = ctypes.c_size_t(0)
    _check("fl_moe_int4g_workspace",
           lib().fl_moe_int4g_workspace(M, E, k, H, I, int(bool(has_shared)), ctypes.byref(out)))
    return out.value


def fl_moe_int4g(x, logits, k, I, w13, w2, scoring=FL_SOFTMAX, renorm=True, shared_w13=None, shared_w2=None,
                 y=None, topk_ids=None, topk_w=None, expert_offsets=None, perm=None, ws=None,
                 score_bias=None, n_group=1, topk_group=1, routed_scale=1.0, group=GROUP):
    """Routed MoE layer.  w13 / w2: uint8 CUDA tensors holding the E
    interleaved expert matrices back to back.  Optional routing outputs are
    written when given.  score_bias (fp32 [E] CUDA tensor), n_group /
    topk_group and routed_scale are the routing options of fl_moe_int4g_ex;
    with their defaults this is fl_moe_int4g."""
    torch = _torch()
    M, H = x.shape
    E = logits.shape[1]
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    has_shared = shared_w13 is not None
    nb = fl_moe_int4g_workspace(M, E, k, H, I, has_shared)
    if ws is None:
        ws = _workspace(nb, x.device)
    if group != GROUP:
        r = FlMoeRouting(scoring, int(bool(renorm)), _p(score_bias), int(n_group), int(topk_group),
                         float(routed_scale))
        _check("fl_moe_int4g_g",
               lib().fl_moe_int4g_g(_p(x), _p(logits), M, H, E, k, I, ctypes.byref(r), int(group),
                                    _p(w13), _p(w2), _p(shared_w13), _p(shared_w2), _p(y),
                                    _p(topk_ids), _p(topk_w), _p(expert_offsets), _p(perm),
                                    _p(ws), ws.numel(), _stream()))
        return y
    if score_bias is None and n_group <= 1 and routed_scale == 1.0:
        _check("fl_moe_int4g",
               lib().fl_moe_int4g(_p(x), _p(logits), M, H, E, k, I, scoring, int(bool(renorm)),
                                  _p(w13), _p(w2), _p(shared_w13), _p(shared_w2), _p(y),
                                  _p(topk_ids), _p(topk_w), _p(expert_offsets), _p(perm),
                                  _p(ws), ws.numel(), _stream()))
        return y
    r = FlMoeRouting(scoring, int(bool(renorm)), _p(score_bias), int(n_group), int(topk_group), float(routed_scale))
    _check("fl_moe_int4g_ex",
           lib().fl_moe_int4g_ex(_p(x), _p(logits), M, H, E, k, I, ctypes.byref(r),
                                 _p(w13), _p(w2), _p(shared_w13), _p(shared_w2), _p(y),
                                 _p(topk_ids), _p(topk_w), _p(expert_offsets), _p(perm),
                                 _p(ws), ws.numel(), _stream()))
    return y


def fl_moe_int4g_ptrs(x, logits, k, I, w13_list, w2_list, scoring=FL_SOFTMAX, renorm=True, shared_w13=None,
                      shared_w2=None, y=None, topk_ids=None, topk_w=None, expert_offsets=None, perm=None, ws=None,
                      score_bias=None, n_group=1, topk_group=1, routed_scale=1.0, tables=None):
    """Routed MoE layer with each expert's matrices in its own CUDA tensor
    (w13_list[e]: interleaved [2I, H], w2_list[e]: interleaved [H, I]).  The
    device tables of expert pointers are built here (int64 CUDA tensors) or
    taken from `tables` = (w13_table, w2_table) when given."""
    torch = _torch()
    M, H = x.shape
    E = logits.shape[1]
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    if tables is None:
        tables = (torch.tensor([t.data_ptr() for t in w13_list], dtype=torch.int64, device=x.device),
                  torch.tensor([t.data_ptr() for t in w2_list], dtype=torch.int64, device=x.device))
    nb = fl_moe_int4g_workspace(M, E, k, H, I, shared_w13 is not None)
    if ws is None:
        ws = _workspace(nb, x.device)
    r = FlMoeRouting(scoring, int(bool(renorm)), _p(score_bias), int(n_group), int(topk_group), float(routed_scale))
    _check("fl_moe_int4g_ptrs",
           lib().fl_moe_int4g_ptrs(_p(x), _p(logits), M, H, E, k, I, ctypes.byref(r),
                                   _p(tables[0]), _p(tables[1]), _p(shared_w13), _p(shared_w2), _p(y),
                                   _p(topk_ids), _p(topk_w), _p(expert_offsets), _p(perm),
                                   _p(ws), ws.numel(), _stream()))
    return y


def fl_moe_router_logits_workspace(M, H, E):
    out = ctypes.c_size_t(0)
    _check("fl_moe_router_logits_workspace", lib().fl_moe_router_logits_workspace(M, H, E, ctypes.byref(out)))
    return out.value


def fl_moe_router_logits(x, w_router, logits=None, ws=None):
    """fp32 [M, E] router logits = x[M, H] . w_router[E, H]^T (bf16 inputs)."""
    torch = _torch()
    M, H = x.shape
    E = w_router.shape[0]
    if logits is None:
        logits = torch.empty((M, E), dtype=torch.float32, device=x.device)
    nb = fl_moe_router_logits_workspace(M, H, E)
    if ws is None:
        ws = _workspace(nb, x.device)
    _check("fl_moe_router_logits", lib().fl_moe_router_logits(_p(x), M, H, _p(w_router), E, _p(logits), _p(ws),
                                                               ws.numel(), _stream()))
    return logits
