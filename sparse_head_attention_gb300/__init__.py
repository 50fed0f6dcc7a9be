"""Elastic Attention hybrid-head attention on GB300 (sm_103a).

Thin Python binding over the C ABI declared in ``include/ea.h``; the names match
the C entry points.  This module only marshals arguments (pointers, strides,
streams) from torch tensors: every step of the computation runs in the CUDA
library ``_lib/libea.so``.  If that library is missing, or no CUDA device is
present, the device entry points raise instead of computing anything else.

    ea_route                 router pre-pass (pool -> MLP -> argmax -> mode)
    ea_route_layers          the router pre-pass of many model layers in one launch
    ea_hybrid_attn_prefill   fused FA / SSA / block-sparse prefill, one launch
    ea_hybrid_attn_prefill_host  the prefill on host tensors, copies overlapped
    ea_hybrid_attn_prefill_varlen  sequences of different lengths in one launch
    ea_hybrid_attn_decode    split-KV decode with the prefill-time routing
    ea_hybrid_attn_decode_paged  the same decode over a paged KV cache
    ea_sparsity_ratios       Omega_MSR / Omega_ESR (host)
    ea_check_errors          read back the device error word of a workspace
"""
import ctypes
import math
import os

import torch

FULL, SSA, BLOCK = 0, 1, 2
TILE = 128
EA_OK = 0
_STATUS = {0: "EA_OK", 1: "EA_ERR_INVALID_ARG", 2: "EA_ERR_UNSUPPORTED", 3: "EA_ERR_WORKSPACE",
           4: "EA_ERR_CUDA", 5: "EA_ERR_TIMEOUT", 6: "EA_ERR_DEVICE_CHECK"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libea.so")
_lib = None

# Function names exported by the library (the ones include/ea.h declares).
EXPORTS = ("ea_status_string", "ea_route", "ea_route_layers", "ea_prefill_workspace_size", "ea_hybrid_attn_prefill",
           "ea_prefill_plan", "ea_prefill_attend", "ea_hybrid_attn_prefill_noalloc",
           "ea_prefill_host_buffer_size", "ea_hybrid_attn_prefill_host",
           "ea_prefill_varlen_workspace_size", "ea_hybrid_attn_prefill_varlen",
           "ea_prefill_layers_workspace_size", "ea_hybrid_attn_prefill_layers",
           "ea_decode_workspace_size",
           "ea_hybrid_attn_decode", "ea_hybrid_attn_decode_paged", "ea_xa_workspace_size",
           "ea_xa_estimate", "ea_sparsity_ratios", "ea_check_errors")


class EAError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, _STATUS.get(status, status)))


class _Mlp(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("dims", ctypes.POINTER(ctypes.c_int)),
                ("W", ctypes.POINTER(ctypes.c_void_p)), ("b", ctypes.POINTER(ctypes.c_void_p))]


class _PrefillLayer(ctypes.Structure):
    _fields_ = [("Q", ctypes.c_void_p), ("K", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("O", ctypes.c_void_p), ("LSE", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("block_mask", ctypes.c_void_p)]


MAX_PREFILL_LAYERS = 48


class _Policy(ctypes.Structure):
    _fields_ = [("fa_impl", ctypes.c_uint8), ("sa_impl", ctypes.c_uint8)]


def use_library(path):
    """Route every later call through the library at `path` (for example the
    bounds-checked build, _lib/libea_checked.so); returns the previous path."""
    global _lib, LIB_PATH
    prev = LIB_PATH
    LIB_PATH = path
    _lib = None
    return prev


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libea.so is not built; run __graft_entry__.build() or "
                               "python sparse_head_attention_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, sz, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float,
                                ctypes.c_double)
        L.ea_status_string.argtypes = [i32]
        L.ea_status_string.restype = ctypes.c_char_p
        L.ea_route.argtypes = [P, P, i32, i32, i32, i32, i32, i32, ctypes.POINTER(_Mlp), _Policy,
                               P, P, P, P]
        L.ea_route_layers.argtypes = [P, i32, P, i32, i32, i32, i32, i32, i32, P, _Policy,
                                      P, P, P, P]
        L.ea_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.ea_prefill_workspace_size.restype = sz
        L.ea_hybrid_attn_prefill.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                             P, i32, i32, P, i32, P, sz, P, P]
        L.ea_prefill_plan.argtypes = [i32, i32, i32, i32, i32, P, i32, i32, P, i32, P, sz, P]
        L.ea_prefill_attend.argtypes = list(L.ea_hybrid_attn_prefill.argtypes)
        L.ea_hybrid_attn_prefill_noalloc.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                     i32, f32, P, i32, i32, P, i32, P, P]
        L.ea_hybrid_attn_prefill_noalloc.restype = ctypes.c_int
        L.ea_prefill_host_buffer_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.ea_prefill_host_buffer_size.restype = sz
        L.ea_hybrid_attn_prefill_host.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, f32, P,
                                                  i32, i32, P, i32, P, sz, i32, P]
        L.ea_hybrid_attn_prefill_host.restype = ctypes.c_int
        L.ea_prefill_layers_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.ea_prefill_layers_workspace_size.restype = sz
        L.ea_hybrid_attn_prefill_layers.argtypes = [P, i32, P, P, P, i32, i32, i32, i32, i32, f32,
                                                    i32, i32, i32, P, sz, P]
        L.ea_hybrid_attn_prefill_layers.restype = ctypes.c_int
        L.ea_prefill_varlen_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.ea_prefill_varlen_workspace_size.restype = sz
        L.ea_hybrid_attn_prefill_varlen.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                    i32, i32, f32, P, i32, i32, P, i32, P, sz, P]
        L.ea_hybrid_attn_prefill_varlen.restype = ctypes.c_int
        L.ea_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.ea_decode_workspace_size.restype = sz
        L.ea_hybrid_attn_decode.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, f32,
                                            P, i32, i32, P, i32, i32, P, sz, P]
        L.ea_hybrid_attn_decode_paged.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_int64, i32,
                                                  i32, i32, P, i32, i32, i32, i32, f32, P, i32,
                                                  i32, P, i32, i32, P, sz, P]
        L.ea_hybrid_attn_decode_paged.restype = ctypes.c_int
        L.ea_xa_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        L.ea_xa_workspace_size.restype = sz
        L.ea_xa_estimate.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, P, i32, f32, i32,
                                     i32, P, P, P, sz, P]
        L.ea_xa_estimate.restype = ctypes.c_int
        L.ea_sparsity_ratios.argtypes = [P, P, i32, i32, i32, i32, i32, P, i32,
                                         ctypes.POINTER(f64), ctypes.POINTER(f64)]
        L.ea_check_errors.argtypes = [P, P]
        for f in ("ea_route", "ea_route_layers", "ea_hybrid_attn_prefill", "ea_prefill_plan", "ea_prefill_attend",
                  "ea_hybrid_attn_decode",
                  "ea_sparsity_ratios", "ea_check_errors"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(fn, status):
    if status != EA_OK:
        raise EAError(fn, status)


def _dev(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _strides(t):
    return (ctypes.c_int64 * t.dim())(*t.stride())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _mlp_struct(weights, biases):
    """(ea_mlp, keep-alive list) for float32 CUDA weights [out, in] and biases [out]."""
    Ws = [_dev(w, "W", torch.float32).contiguous() for w in weights]
    bs = [_dev(b, "b", torch.float32).contiguous() for b in biases]
    dims = [Ws[0].shape[1]] + [w.shape[0] for w in Ws]
    c_dims = (ctypes.c_int * len(dims))(*dims)
    c_W = (ctypes.c_void_p * len(Ws))(*[w.data_ptr() for w in Ws])
    c_b = (ctypes.c_void_p * len(bs))(*[b.data_ptr() for b in bs])
    return _Mlp(len(Ws), c_dims, c_W, c_b), [Ws, bs, c_dims, c_W, c_b]


def ea_route(K, weights, biases, *, pool_head=100, pool_tail=100, policy=(FULL, SSA),
             r_out=None, m_out=None, logits_out=None, stream=None):
    """Router pre-pass on K [B, S, Hkv, d] (bf16, CUDA).  weights/biases: lists of
    float32 CUDA tensors ([out, in] and [out]).  Returns (r, m, logits)."""
    _dev(K, "K", torch.bfloat16)
    B, S, Hkv, d = K.shape
    dev = K.device
    r_out = r_out if r_out is not None else torch.empty(B, Hkv, dtype=torch.uint8, device=dev)
    m_out = m_out if m_out is not None else torch.empty(B, Hkv, dtype=torch.uint8, device=dev)
    if logits_out is None:
        logits_out = torch.empty(B, Hkv, 2, dtype=torch.float64, device=dev)
    mlp, _keep = _mlp_struct(weights, biases)
    st = lib().ea_route(_ptr(K), _strides(K), B, S, Hkv, d, pool_head, pool_tail,
                        ctypes.byref(mlp), _Policy(*policy), _ptr(r_out), _ptr(m_out),
                        _ptr(logits_out), _stream(stream))
    _check("ea_route", st)
    return r_out, m_out, logits_out


def ea_route_layers(K_layers, weights, biases, *, pool_head=100, pool_tail=100,
                    policy=(FULL, SSA), r_out=None, m_out=None, logits_out=None, stream=None):
    """Router pre-pass of L layers at once.  K_layers: L bf16 CUDA tensors
    [B, S, Hkv, d] with equal shapes and strides; weights[l] / biases[l]: layer
    l's MLP as for ea_route.  Returns (r [L, B, Hkv], m [L, B, Hkv],
    logits [L, B, Hkv, 2])."""
    L = len(K_layers)
    if L < 1 or len(weights) != L or len(biases) != L:
        raise ValueError("K_layers, weights and biases need one entry per layer")
    K0 = _dev(K_layers[0], "K", torch.bfloat16)
    for K in K_layers:
        _dev(K, "K", torch.bfloat16)
        if K.shape != K0.shape or K.stride() != K0.stride():
            raise ValueError("every layer's K needs the same shape and strides")
    B, S, Hkv, d = K0.shape
    dev = K0.device
    if r_out is None:
        r_out = torch.empty(L, B, Hkv, dtype=torch.uint8, device=dev)
    if m_out is None:
        m_out = torch.empty(L, B, Hkv, dtype=torch.uint8, device=dev)
    if logits_out is None:
        logits_out = torch.empty(L, B, Hkv, 2, dtype=torch.float64, device=dev)
    built = [_mlp_struct(w, b) for w, b in zip(weights, biases)]
    mlps = (_Mlp * L)(*[m for m, _ in built])
    ptrs = (ctypes.c_void_p * L)(*[K.data_ptr() for K in K_layers])
    st = lib().ea_route_layers(ptrs, L, _strides(K0), B, S, Hkv, d, pool_head, pool_tail, mlps,
                               _Policy(*policy), _ptr(r_out), _ptr(m_out), _ptr(logits_out),
                               _stream(stream))
    _check("ea_route_layers", st)
    return r_out, m_out, logits_out


def ea_prefill_workspace_size(B, S, Hq, Hkv, d=128):
    return int(lib().ea_prefill_workspace_size(B, S, Hq, Hkv, d))


def prefill_workspace(B, S, Hq, Hkv, d=128, device="cuda"):
    """A zeroed workspace buffer of the right size (256-byte aligned by torch)."""
    n = ea_prefill_workspace_size(B, S, Hq, Hkv, d)
    if n == 0:
        raise ValueError("unsupported prefill sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ea_hybrid_attn_prefill(Q, K, V, m, *, sink, window, block_mask=None, scale=None, O=None,
                           LSE=None, workspace=None, visited_bitmap=None, stream=None,
                           want_lse=True, _entry="ea_hybrid_attn_prefill"):
    """Fused hybrid-head prefill.  Q [B, S, Hq, d], K/V [B, S, Hkv, d] bf16 (CUDA),
    m uint8 [B, Hkv] (CUDA).  Returns (O, LSE)."""
    _dev(Q, "Q", torch.bfloat16)
    _dev(K, "K", torch.bfloat16)
    _dev(V, "V", torch.bfloat16)
    _dev(m, "m", torch.uint8)
    if K.stride() != V.stride():
        raise ValueError("K and V must share strides")
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None and want_lse:
        LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=Q.device)
    if workspace is None:
        workspace = prefill_workspace(B, S, Hq, Hkv, d, Q.device)
    if block_mask is not None:
        _dev(block_mask, "block_mask", torch.uint8)
        if not block_mask.is_contiguous():
            raise ValueError("block_mask must be contiguous")
    st = getattr(lib(), _entry)(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _strides(Q), _strides(K), _strides(O),
        B, S, Hq, Hkv, d, float(scale), _ptr(m), int(sink), int(window), _ptr(block_mask), TILE,
        _ptr(workspace), workspace.numel(), _ptr(visited_bitmap), _stream(stream))
    _check(_entry, st)
    return O, LSE


def ea_prefill_plan(B, S, Hq, Hkv, m, *, sink, window, block_mask=None, workspace, d=128,
                    stream=None):
    """Enqueue the planner only (work queue into `workspace`)."""
    _dev(m, "m", torch.uint8)
    st = lib().ea_prefill_plan(B, S, Hq, Hkv, d, _ptr(m), int(sink), int(window), _ptr(block_mask),
                               TILE, _ptr(workspace), workspace.numel(), _stream(stream))
    _check("ea_prefill_plan", st)


def ea_prefill_attend(Q, K, V, m, *, sink, window, workspace, **kw):
    """Enqueue the attention kernel on a plan made by ea_prefill_plan."""
    return ea_hybrid_attn_prefill(Q, K, V, m, sink=sink, window=window, workspace=workspace,
                                  _entry="ea_prefill_attend", **kw)


def ea_hybrid_attn_prefill_noalloc(Q, K, V, m, *, sink, window, block_mask=None, scale=None,
                                   O=None, LSE=None, visited_bitmap=None, stream=None,
                                   want_lse=True):
    """ea_hybrid_attn_prefill without a workspace, for callers that cannot
    allocate device memory for the library: the planner's scratch is a fixed
    4 MiB array inside it, shared by every call (calls that overlap on the GPU
    race).  Returns (O, LSE)."""
    _dev(Q, "Q", torch.bfloat16)
    _dev(K, "K", torch.bfloat16)
    _dev(V, "V", torch.bfloat16)
    _dev(m, "m", torch.uint8)
    if K.stride() != V.stride():
        raise ValueError("K and V must share strides")
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None and want_lse:
        LSE = torch.empty(B, Hq, S, dtype=torch.float32, device=Q.device)
    if block_mask is not None:
        _dev(block_mask, "block_mask", torch.uint8)
        if not block_mask.is_contiguous():
            raise ValueError("block_mask must be contiguous")
    st = lib().ea_hybrid_attn_prefill_noalloc(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _strides(Q), _strides(K), _strides(O),
        B, S, Hq, Hkv, d, float(scale), _ptr(m), int(sink), int(window), _ptr(block_mask), TILE,
        _ptr(visited_bitmap), _stream(stream))
    _check("ea_hybrid_attn_prefill_noalloc", st)
    return O, LSE


def ea_prefill_layers_workspace_size(n_layers, B, S, Hq, Hkv, d=128):
    return int(lib().ea_prefill_layers_workspace_size(n_layers, B, S, Hq, Hkv, d))


def prefill_layers_workspace(n_layers, B, S, Hq, Hkv, d=128, device="cuda"):
    n = ea_prefill_layers_workspace_size(n_layers, B, S, Hq, Hkv, d)
    if n == 0:
        raise ValueError("unsupported multi-layer prefill sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ea_hybrid_attn_prefill_layers(Qs, Ks, Vs, ms, *, sink, window, block_masks=None, scale=None,
                                  Os=None, LSEs=None, workspace=None, stream=None, want_lse=True):
    """Several layers (same shapes and strides) in one planner + one launch.
    Qs/Ks/Vs/ms: lists of per-layer CUDA tensors as for ea_hybrid_attn_prefill;
    block_masks: None or a list (entries may be None).  Returns (Os, LSEs)."""
    L = len(Qs)
    if not (len(Ks) == len(Vs) == len(ms) == L) or L < 1:
        raise ValueError("one Q, K, V and m per layer")
    for t, nm in ((Qs, "Q"), (Ks, "K"), (Vs, "V")):
        for x in t:
            _dev(x, nm, torch.bfloat16)
    for x in ms:
        _dev(x, "m", torch.uint8)
    B, S, Hq, d = Qs[0].shape
    Hkv = Ks[0].shape[2]
    for l in range(L):
        if (Qs[l].shape != Qs[0].shape or Ks[l].shape != Ks[0].shape or Vs[l].shape != Ks[0].shape or
                Qs[l].stride() != Qs[0].stride() or Ks[l].stride() != Ks[0].stride() or
                Vs[l].stride() != Ks[0].stride()):
            raise ValueError("every layer must have the same shapes and strides")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if Os is None:
        Os = [torch.empty_like(Qs[0]) for _ in range(L)]
    if LSEs is None:
        LSEs = [torch.empty(B, Hq, S, dtype=torch.float32, device=Qs[0].device) if want_lse else None
                for _ in range(L)]
    bms = list(block_masks) if block_masks is not None else [None] * L
    for bm in bms:
        if bm is not None:
            _dev(bm, "block_mask", torch.uint8)
            if not bm.is_contiguous():
                raise ValueError("block_mask must be contiguous")
    if workspace is None:
        workspace = prefill_layers_workspace(L, B, S, Hq, Hkv, d, Qs[0].device)
    arr = (_PrefillLayer * L)()
    for l in range(L):
        arr[l] = _PrefillLayer(Qs[l].data_ptr(), Ks[l].data_ptr(), Vs[l].data_ptr(), Os[l].data_ptr(),
                               LSEs[l].data_ptr() if LSEs[l] is not None else None, ms[l].data_ptr(),
                               bms[l].data_ptr() if bms[l] is not None else None)
    st = lib().ea_hybrid_attn_prefill_layers(
        ctypes.cast(arr, ctypes.c_void_p), L, _strides(Qs[0]), _strides(Ks[0]), _strides(Os[0]), B, S,
        Hq, Hkv, d, float(scale), int(sink), int(window), TILE, _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check("ea_hybrid_attn_prefill_layers", st)
    return Os, LSEs


def ea_prefill_host_buffer_size(B, S, Hq, Hkv, d=128, with_block_mask=False):
    return int(lib().ea_prefill_host_buffer_size(B, S, Hq, Hkv, d, 1 if with_block_mask else 0))


def prefill_host_buffer(B, S, Hq, Hkv, d=128, with_block_mask=False, device="cuda"):
    """Device scratch for ea_hybrid_attn_prefill_host (256-byte aligned by torch)."""
    n = ea_prefill_host_buffer_size(B, S, Hq, Hkv, d, with_block_mask)
    if n == 0:
        raise ValueError("unsupported prefill sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _host(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous host %s tensor" % (name, dtype))
    return t


def ea_hybrid_attn_prefill_host(Q, K, V, m, *, sink, window, block_mask=None, scale=None, O=None,
                                LSE=None, device_buffer=None, n_chunks=0, stream=None,
                                want_lse=True):
    """The fused prefill on HOST tensors (contiguous; page-locked for overlap):
    Q [B, S, Hq, d], K/V [B, S, Hkv, d] bf16, m uint8 [B, Hkv], block_mask uint8
    [B, Hkv, nB, nB] or None.  Copies in, attention and copies out run as a
    chunked pipeline on the current CUDA device.  Returns (O, LSE) as host
    tensors, complete once `stream` (default: the current stream) has passed
    the call's work."""
    _host(Q, "Q", torch.bfloat16)
    _host(K, "K", torch.bfloat16)
    _host(V, "V", torch.bfloat16)
    _host(m, "m", torch.uint8)
    if block_mask is not None:
        _host(block_mask, "block_mask", torch.uint8)
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = Q.is_pinned()
    if O is None:
        O = torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=pin)
    _host(O, "O", torch.bfloat16)
    if LSE is None and want_lse:
        LSE = torch.empty(B, Hq, S, dtype=torch.float32, pin_memory=pin)
    if LSE is not None:
        _host(LSE, "LSE", torch.float32)
    if device_buffer is None:
        device_buffer = prefill_host_buffer(B, S, Hq, Hkv, d, block_mask is not None)
    _dev(device_buffer, "device_buffer", torch.uint8)
    st = lib().ea_hybrid_attn_prefill_host(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, S, Hq, Hkv, d, float(scale), _ptr(m),
        int(sink), int(window), _ptr(block_mask), TILE, _ptr(device_buffer),
        device_buffer.numel(), int(n_chunks), _stream(stream))
    _check("ea_hybrid_attn_prefill_host", st)
    return O, LSE


def ea_prefill_varlen_workspace_size(B, total_tokens, max_seqlen, Hq, Hkv, d=128):
    return int(lib().ea_prefill_varlen_workspace_size(B, total_tokens, max_seqlen, Hq, Hkv, d))


def prefill_varlen_workspace(B, total_tokens, max_seqlen, Hq, Hkv, d=128, device="cuda"):
    n = ea_prefill_varlen_workspace_size(B, total_tokens, max_seqlen, Hq, Hkv, d)
    if n == 0:
        raise ValueError("unsupported variable-length prefill sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ea_hybrid_attn_prefill_varlen(Q, K, V, cu_seqlens, m, *, max_seqlen, sink, window,
                                  block_mask=None, scale=None, O=None, LSE=None, workspace=None,
                                  stream=None, want_lse=True):
    """Sequences of different lengths packed back to back, one launch.
    Q [total, Hq, d], K/V [total, Hkv, d] bf16; cu_seqlens int32 [B + 1];
    m uint8 [B, Hkv]; block_mask uint8, per sequence [Hkv, nB_b, nB_b] back
    to back (or None); all CUDA.  Returns (O [total, Hq, d], LSE [Hq, total])."""
    _dev(Q, "Q", torch.bfloat16)
    _dev(K, "K", torch.bfloat16)
    _dev(V, "V", torch.bfloat16)
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(m, "m", torch.uint8)
    if K.stride() != V.stride():
        raise ValueError("K and V must share strides")
    total, Hq, d = Q.shape
    Hkv = K.shape[1]
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None and want_lse:
        LSE = torch.empty(Hq, total, dtype=torch.float32, device=Q.device)
    if workspace is None:
        workspace = prefill_varlen_workspace(B, total, max_seqlen, Hq, Hkv, d, Q.device)
    st = lib().ea_hybrid_attn_prefill_varlen(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _strides(Q), _strides(K), _strides(O),
        _ptr(cu_seqlens), B, total, int(max_seqlen), Hq, Hkv, d, float(scale), _ptr(m), int(sink),
        int(window), _ptr(block_mask), TILE, _ptr(workspace), workspace.numel(), _stream(stream))
    _check("ea_hybrid_attn_prefill_varlen", st)
    return O, LSE


def ea_decode_workspace_size(B, Hq, Hkv, Lmax, num_splits=0, d=128):
    return int(lib().ea_decode_workspace_size(B, Hq, Hkv, d, Lmax, num_splits))


def decode_workspace(B, Hq, Hkv, Lmax, num_splits=0, d=128, device="cuda"):
    n = ea_decode_workspace_size(B, Hq, Hkv, Lmax, num_splits, d)
    if n == 0:
        raise ValueError("unsupported decode sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _block_mask_arg(block_mask, B, Hkv, Lmax):
    if block_mask is None:
        return None
    _dev(block_mask, "block_mask", torch.uint8)
    nB = (Lmax + TILE - 1) // TILE
    if tuple(block_mask.shape) != (B, Hkv, nB, nB) or not block_mask.is_contiguous():
        raise ValueError("block_mask must be a contiguous [B, Hkv, %d, %d] tensor" % (nB, nB))
    return block_mask


def ea_hybrid_attn_decode(q, Kc, Vc, seqlens, m, *, sink, window, block_mask=None, num_splits=0,
                          scale=None, O=None, LSE=None, workspace=None, stream=None, want_lse=True):
    """One decode step.  q [B, Hq, d], Kc/Vc [B, Lmax, Hkv, d] bf16 (CUDA),
    seqlens int32 [B] (CUDA), m uint8 [B, Hkv] (CUDA), block_mask uint8
    [B, Hkv, nB, nB] (nB = ceil(Lmax / 128), CUDA) when a head is BLOCK.
    Returns (O, LSE)."""
    _dev(q, "q", torch.bfloat16)
    _dev(Kc, "Kc", torch.bfloat16)
    _dev(Vc, "Vc", torch.bfloat16)
    _dev(seqlens, "seqlens", torch.int32)
    _dev(m, "m", torch.uint8)
    if Kc.stride() != Vc.stride():
        raise ValueError("Kc and Vc must share strides")
    B, Hq, d = q.shape
    Lmax, Hkv = Kc.shape[1], Kc.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(q)
    if LSE is None and want_lse:
        LSE = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, Lmax, num_splits, d, q.device)
    bm = _block_mask_arg(block_mask, B, Hkv, Lmax)
    st = lib().ea_hybrid_attn_decode(
        _ptr(q), _ptr(Kc), _ptr(Vc), _ptr(O), _ptr(LSE), _strides(q), _strides(Kc), _strides(O),
        _ptr(seqlens), B, Hq, Hkv, d, Lmax, float(scale), _ptr(m), int(sink), int(window),
        _ptr(bm), TILE, int(num_splits), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("ea_hybrid_attn_decode", st)
    return O, LSE


def ea_hybrid_attn_decode_paged(q, K_pages, V_pages, block_table, seqlens, m, *, sink, window,
                                block_mask=None, num_splits=0, scale=None, O=None, LSE=None,
                                workspace=None, stream=None, want_lse=True):
    """One decode step over a paged cache.  q [B, Hq, d]; K_pages/V_pages
    [num_pages, page_size, Hkv, d] bf16; block_table int32 [B, max_pages] (key
    k of sequence b: row k % page_size of page block_table[b, k // page_size]);
    seqlens int32 [B]; m uint8 [B, Hkv]; all CUDA.  Returns (O, LSE)."""
    _dev(q, "q", torch.bfloat16)
    _dev(K_pages, "K_pages", torch.bfloat16)
    _dev(V_pages, "V_pages", torch.bfloat16)
    _dev(block_table, "block_table", torch.int32)
    _dev(seqlens, "seqlens", torch.int32)
    _dev(m, "m", torch.uint8)
    if K_pages.stride() != V_pages.stride() or K_pages.shape != V_pages.shape:
        raise ValueError("K_pages and V_pages must share shapes and strides")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [B, max_pages] with unit column stride")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv = K_pages.shape[0], K_pages.shape[1], K_pages.shape[2]
    max_pages = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if O is None:
        O = torch.empty_like(q)
    if LSE is None and want_lse:
        LSE = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, max_pages * page_size, num_splits, d, q.device)
    bm = _block_mask_arg(block_mask, B, Hkv, max_pages * page_size)
    st = lib().ea_hybrid_attn_decode_paged(
        _ptr(q), _ptr(K_pages), _ptr(V_pages), _ptr(O), _ptr(LSE), _strides(q), _strides(K_pages),
        _strides(O), _ptr(block_table), block_table.stride(0), max_pages, page_size, num_pages,
        _ptr(seqlens), B, Hq, Hkv, d, float(scale), _ptr(m), int(sink), int(window),
        _ptr(bm), TILE, int(num_splits), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("ea_hybrid_attn_decode_paged", st)
    return O, LSE


XA_STRIDE = 16


def ea_xa_workspace_size(B, S, Hq, Hkv, max_units, d=128, stride=XA_STRIDE):
    return int(lib().ea_xa_workspace_size(B, S, Hq, Hkv, d, stride, max_units))


def xa_workspace(B, S, Hq, Hkv, max_units, d=128, device="cuda"):
    """A zeroed XA estimation workspace for at most max_units BLOCK (b, KV head) units."""
    n = ea_xa_workspace_size(B, S, Hq, Hkv, max_units, d)
    if n == 0:
        raise ValueError("unsupported XA estimation sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ea_xa_estimate(Q, K, m, *, threshold=0.9, max_units=None, block_mask=None,
                   block_scores=None, want_scores=False, scale=None, workspace=None,
                   stride=XA_STRIDE, stream=None):
    """XA block-mask estimation (antidiagonal scoring) for the heads whose mode is
    BLOCK.  Q [B, S, Hq, d], K [B, S, Hkv, d] bf16 (CUDA), m uint8 [B, Hkv] (CUDA).
    Returns (block_mask uint8 [B, Hkv, nB, nB], block_scores float32 or None); rows
    of other heads are left as they are in a caller-given block_mask (zeros in a
    new one)."""
    _dev(Q, "Q", torch.bfloat16)
    _dev(K, "K", torch.bfloat16)
    _dev(m, "m", torch.uint8)
    B, S, Hq, d = Q.shape
    Hkv = K.shape[2]
    nB = (S + TILE - 1) // TILE
    if max_units is None:
        max_units = B * Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if block_mask is None:
        block_mask = torch.zeros(B, Hkv, nB, nB, dtype=torch.uint8, device=Q.device)
    _dev(block_mask, "block_mask", torch.uint8)
    if not block_mask.is_contiguous():
        raise ValueError("block_mask must be contiguous")
    if block_scores is None and want_scores:
        block_scores = torch.zeros(B, Hkv, nB, nB, dtype=torch.float32, device=Q.device)
    if block_scores is not None:
        _dev(block_scores, "block_scores", torch.float32)
        if not block_scores.is_contiguous():
            raise ValueError("block_scores must be contiguous")
    if workspace is None:
        workspace = xa_workspace(B, S, Hq, Hkv, max_units, d, Q.device)
    st = lib().ea_xa_estimate(_ptr(Q), _ptr(K), _strides(Q), _strides(K), B, S, Hq, Hkv, d,
                              float(scale), _ptr(m), int(stride), float(threshold), TILE,
                              int(max_units), _ptr(block_mask), _ptr(block_scores),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check("ea_xa_estimate", st)
    return block_mask, block_scores


def ea_sparsity_ratios(r, m, S, *, sink, window, block_masks=None):
    """Host: (Omega_MSR, Omega_ESR) for r, m uint8 [L, Hkv] (CPU tensors or arrays);
    block_masks: None or a list of L uint8 [Hkv, nB, nB] CPU arrays (None entries
    for layers without BLOCK heads)."""
    import numpy as np
    ra = np.ascontiguousarray(np.asarray(r.cpu() if isinstance(r, torch.Tensor) else r), np.uint8)
    ma = np.ascontiguousarray(np.asarray(m.cpu() if isinstance(m, torch.Tensor) else m), np.uint8)
    L, Hkv = ra.shape
    keep = []
    c_masks = None
    if block_masks is not None:
        c_masks = (ctypes.c_void_p * L)()
        for l, bm in enumerate(block_masks):
            if bm is None:
                c_masks[l] = None
                continue
            a = np.ascontiguousarray(np.asarray(bm.cpu() if isinstance(bm, torch.Tensor) else bm),
                                     np.uint8)
            keep.append(a)
            c_masks[l] = a.ctypes.data
    msr, esr = ctypes.c_double(), ctypes.c_double()
    st = lib().ea_sparsity_ratios(ra.ctypes.data, ma.ctypes.data, L, Hkv, S, sink, window,
                                  c_masks, TILE, ctypes.byref(msr), ctypes.byref(esr))
    _check("ea_sparsity_ratios", st)
    return msr.value, esr.value


def ea_check_errors(workspace, stream=None):
    """Synchronise and read/clear the device error word; returns the status code."""
    return lib().ea_check_errors(_ptr(workspace), _stream(stream))
