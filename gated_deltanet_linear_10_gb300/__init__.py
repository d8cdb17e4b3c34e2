"""Python binding of libgdn, the GB300 Gated DeltaNet layer library.

Each function below has the name of a C entry point declared in
``include/gdn.h`` and only marshals arguments: it checks shapes, dtypes and
devices of PyTorch tensors, allocates the outputs that were not passed (with
PyTorch), and calls the C ABI on the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no other path.  If
``libgdn.so`` is not built, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

(GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_LAUNCH, GDN_ERR_CUDA,
 GDN_ERR_TOO_LARGE) = range(6)
PREFILL_STATIC_SCRATCH_BYTES = 16 << 20
GDN_F32, GDN_BF16 = 0, 1
DEVSTAT_BAD_INDEX, DEVSTAT_BAD_SEQLEN, DEVSTAT_TIMEOUT = 0x1, 0x2, 0x4

# Every symbol the header declares (checked by the tests against the .so).
EXPORTS = (
    "gdn_status_string", "gdn_version", "gdn_last_cuda_error", "gdn_gating",
    "causal_conv1d_fwd", "causal_conv1d_update", "gdn_prefill_chunked",
    "gdn_prefill_workspace_size", "gdn_decode_recurrent", "gdn_state_snapshot",
    "gdn_get_device_status", "gdn_prefill_chunked_static", "gdn_gated_rmsnorm",
    "gdn_decode_recurrent_gated", "gdn_decode_step_fused", "gdn_mixed_batch",
    "gdn_debug_set_wait_limit", "gdn_prefill_chunked_gated", "gdn_mtp_step_fused",
    "gdn_decode_step_workspace_size", "gdn_prefill_layer", "gdn_prefill_layer_workspace_size",
    "gdn_prefill_layer_gated",
)

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                      f"g.build()'` (nvcc, sm_103a) first")

_lib = ctypes.CDLL(LIB_PATH)

_vp, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_lib.gdn_status_string.restype = ctypes.c_char_p
_lib.gdn_status_string.argtypes = [ctypes.c_int]
_lib.gdn_version.restype = ctypes.c_char_p
_lib.gdn_version.argtypes = []
_lib.gdn_last_cuda_error.restype = ctypes.c_char_p
_lib.gdn_last_cuda_error.argtypes = []
_SIGS = {
    "gdn_gating": [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp, _vp, _vp],
    "causal_conv1d_fwd": [_vp, _i64, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _vp, _i64, _vp, _vp,
                          _i32, _vp, _i32, _vp],
    "causal_conv1d_update": [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp, _i32,
                             _vp, _i32, _vp],
    "gdn_prefill_chunked": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i64, _i32,
                            _i32, _i32, _i32, _f32, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _i32,
                            _vp, ctypes.c_size_t, _vp],
    "gdn_decode_recurrent": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
                             _i32, _i32, _f32, _i32, _vp, _i64, _vp, _vp, _vp, _i32, _vp],
    "gdn_state_snapshot": [_vp, _i64, _i64, _vp, _vp, _i32, _vp],
    "gdn_get_device_status": [ctypes.POINTER(ctypes.c_uint32), _i32, _vp],
    "gdn_decode_step_fused": [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                              _f32, _vp, _i64, _vp, _vp, ctypes.c_size_t, _vp, _vp],
    "gdn_gated_rmsnorm": [_vp, _vp, _i64, _vp, _i64, _i32, _i32, _f32, _vp, _i32, _vp],
    "gdn_decode_recurrent_gated": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _i32, _i32, _i32,
                                   _i32, _i32, _i32, _f32, _i32, _vp, _i64, _vp, _vp, _vp, _i64,
                                   _vp, _f32, _vp, _i32, _vp],
    "gdn_prefill_chunked_static": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i64,
                                   _i32, _i32, _f32, _i32, _vp, _i64, _vp, _vp, _vp, _vp],
    "gdn_debug_set_wait_limit": [ctypes.c_uint64, _i32, _vp],
    "gdn_prefill_layer": [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                          _i64, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _vp,
                          ctypes.c_size_t, _vp],
    "gdn_prefill_layer_gated": [_vp, _i64, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                _i32, _i64, _i32, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _i64, _vp,
                                _f32, _vp, _vp, ctypes.c_size_t, _vp],
    "gdn_mtp_step_fused": [_vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                           _f32, _vp, _i64, _vp, _vp, _vp, _vp],
    "gdn_prefill_chunked_gated": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i64,
                                  _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _i64, _vp, _vp,
                                  _vp, _i64, _vp, _f32, _vp, _i32, _vp, ctypes.c_size_t, _vp],
    "gdn_mixed_batch": [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i64, _i32,
                        _i32, _i32, _i32, _f32, _i32, _i32, _vp, _i64, _vp, _vp, _i32, _vp, _i32,
                        _vp, ctypes.c_size_t, _vp],
}
for _name, _args in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
_lib.gdn_prefill_workspace_size.argtypes = [_i32, _i64, _i32, _i32, _i32, _i32, _i32]
_lib.gdn_prefill_workspace_size.restype = ctypes.c_size_t
_lib.gdn_decode_step_workspace_size.argtypes = [_i32, _i32, _i32]
_lib.gdn_decode_step_workspace_size.restype = ctypes.c_size_t
_lib.gdn_prefill_layer_workspace_size.argtypes = [_i32, _i64, _i32, _i32]
_lib.gdn_prefill_layer_workspace_size.restype = ctypes.c_size_t


class GdnError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != GDN_OK:
        name = _lib.gdn_status_string(status).decode()
        cuda = _lib.gdn_last_cuda_error().decode()
        raise GdnError(f"{what}: {name}" + (f" ({cuda})" if cuda else ""))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDN_F32
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    raise GdnError(f"unsupported activation dtype {t.dtype} (fp32 or bf16)")


def _need(cond: bool, msg: str):
    if not cond:
        raise GdnError(msg)


def _cuda(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda, "all tensors must be on a CUDA device")


def _i32_vec(t, name):
    if t is None:
        return None
    _need(t.dtype == torch.int32 and t.is_contiguous(), f"{name} must be contiguous int32")
    return t


def _heads_view(x, heads, d, name):
    """x is [T, heads, d] (or [T, heads*d]) with unit inner strides; returns row stride."""
    if x.dim() == 2:
        _need(x.shape[1] == heads * d and x.stride(1) == 1, f"{name}: bad shape/stride")
        return x.stride(0)
    _need(x.dim() == 3 and x.shape[1] == heads and x.shape[2] == d, f"{name}: shape {tuple(x.shape)}")
    _need(x.stride(2) == 1 and x.stride(1) == d, f"{name}: heads must be packed ({x.stride()})")
    return x.stride(0)


def version() -> str:
    return _lib.gdn_version().decode()


def gdn_gating(a, b, A_log, dt_bias, g=None, beta=None):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b); a, b: [T, hv]."""
    _cuda(a, b, A_log, dt_bias)
    _need(a.shape == b.shape and a.dim() == 2 and a.dtype == b.dtype, "a, b: [T, hv], same dtype")
    _need(a.is_contiguous() and b.is_contiguous(), "a, b must be contiguous")
    T, hv = a.shape
    _need(A_log.dtype == torch.float32 and dt_bias.dtype == torch.float32, "A_log/dt_bias fp32")
    _need(A_log.numel() == hv and dt_bias.numel() == hv, "A_log/dt_bias: [hv]")
    g = torch.empty((T, hv), dtype=torch.float32, device=a.device) if g is None else g
    beta = torch.empty((T, hv), dtype=torch.float32, device=a.device) if beta is None else beta
    _check(_lib.gdn_gating(_ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), T, hv, _dtype_code(a),
                           _ptr(g), _ptr(beta), _stream(a.device)), "gdn_gating")
    return g, beta


def causal_conv1d_fwd(x, weight, cu_seqlens, conv_state_pool, state_indices,
                      has_initial_state=None, bias=None, silu=True, y=None):
    """Varlen causal conv1d (+SiLU); x [T, C] (row stride free), weight [C, W],
    conv_state_pool [slots, W-1, C]; returns y [T, C]."""
    _cuda(x, weight, cu_seqlens, conv_state_pool, state_indices, has_initial_state, bias)
    _need(x.dim() == 2 and x.stride(1) == 1, "x: [T, C] with unit column stride")
    T, C = x.shape
    _need(weight.shape[0] == C and weight.is_contiguous() and weight.dtype == x.dtype, "weight")
    W = weight.shape[1]
    _need(conv_state_pool.shape[1:] == (W - 1, C) and conv_state_pool.is_contiguous()
          and conv_state_pool.dtype == x.dtype, "conv_state_pool: [slots, W-1, C]")
    _i32_vec(cu_seqlens, "cu_seqlens")
    _i32_vec(state_indices, "state_indices")
    n = cu_seqlens.numel() - 1
    _need(state_indices.numel() == n, "state_indices: [n_seqs]")
    if has_initial_state is not None:
        _need(has_initial_state.dtype == torch.uint8 and has_initial_state.numel() == n,
              "has_initial_state: [n_seqs] uint8")
    y = torch.empty((T, C), dtype=x.dtype, device=x.device) if y is None else y
    _check(_lib.causal_conv1d_fwd(_ptr(x), x.stride(0), _ptr(weight), _ptr(bias), _ptr(cu_seqlens),
                                  n, T, C, W, _ptr(conv_state_pool), conv_state_pool.shape[0],
                                  _ptr(state_indices), _ptr(has_initial_state), int(silu), _ptr(y),
                                  _dtype_code(x), _stream(x.device)), "causal_conv1d_fwd")
    return y


def causal_conv1d_update(x, tokens_per_seq, weight, conv_state_pool, state_indices,
                         snap_indices=None, bias=None, silu=True, y=None):
    """Decode / MTP conv update; x [N*tps, C] contiguous (row i*tps + t)."""
    _cuda(x, weight, conv_state_pool, state_indices, snap_indices, bias)
    _need(x.dim() == 2 and x.is_contiguous(), "x: [N*tps, C] contiguous")
    _i32_vec(state_indices, "state_indices")
    _i32_vec(snap_indices, "snap_indices")
    N = state_indices.numel()
    _need(x.shape[0] == N * tokens_per_seq, "x rows != n_seqs * tokens_per_seq")
    C = x.shape[1]
    W = weight.shape[1]
    _need(conv_state_pool.shape[1:] == (W - 1, C) and conv_state_pool.dtype == x.dtype,
          "conv_state_pool: [slots, W-1, C]")
    if snap_indices is not None:
        _need(snap_indices.numel() == N * tokens_per_seq, "snap_indices: [n_seqs, tps]")
    y = torch.empty_like(x) if y is None else y
    _check(_lib.causal_conv1d_update(_ptr(x), N, tokens_per_seq, C, W, _ptr(weight), _ptr(bias),
                                     _ptr(conv_state_pool), conv_state_pool.shape[0],
                                     _ptr(state_indices), _ptr(snap_indices), int(silu), _ptr(y),
                                     _dtype_code(x), _stream(x.device)), "causal_conv1d_update")
    return y


def gdn_prefill_workspace_size(n_seqs, n_tokens, hv, dk, dv, chunk, dtype=GDN_BF16) -> int:
    return int(_lib.gdn_prefill_workspace_size(n_seqs, n_tokens, hv, dk, dv, chunk, dtype))


def gdn_prefill_chunked(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices,
                        final_state_indices, scale, chunk=64, l2norm_qk=True, o=None,
                        workspace=None):
    """Chunked varlen prefill.  q, k [T, hqk, dk]; v [T, hv, dv] (views with a
    free row stride); g, beta [T, hv] fp32; state_pool [slots, hv, dv, dk]
    fp32.  Returns o [T, hv, dv].

    workspace: None allocates the scratch gdn_prefill_workspace_size asks for
    (the bf16 dk = dv = 128 path then runs as a chunk-parallel prep kernel and
    a chain kernel); a uint8 CUDA tensor is used as given; False passes none,
    which selects the single fused kernel."""
    _cuda(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices, final_state_indices)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v: one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32 and g.is_contiguous()
          and beta.is_contiguous() and g.shape == (T, hv) and beta.shape == (T, hv), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    _i32_vec(cu_seqlens, "cu_seqlens")
    n = cu_seqlens.numel() - 1
    for name, t in (("initial_state_indices", initial_state_indices),
                    ("final_state_indices", final_state_indices)):
        if t is not None:
            _i32_vec(t, name)
            _need(t.numel() == n, f"{name}: [n_seqs]")
    o = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if o is None else o
    _need(o.is_contiguous() and o.shape == (T, hv, dv), "o: [T, hv, dv] contiguous")
    dt = _dtype_code(q)
    if workspace is False:
        workspace = None
    elif workspace is None:
        need = gdn_prefill_workspace_size(n, T, hv, dk, dv, chunk, dt)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    else:
        _cuda(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_prefill_chunked(_ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g), _ptr(beta),
                                    _ptr(cu_seqlens), n, T, hqk, hv, dk, dv, float(scale),
                                    int(l2norm_qk), chunk, _ptr(state_pool), state_pool.shape[0],
                                    _ptr(initial_state_indices), _ptr(final_state_indices),
                                    _ptr(o), dt, _ptr(workspace), wbytes, _stream(q.device)),
           "gdn_prefill_chunked")
    return o


def gdn_prefill_chunked_gated(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices,
                              final_state_indices, scale, z, norm_weight, norm_eps=1e-6, chunk=64,
                              l2norm_qk=True, y=None, workspace=None):
    """gdn_prefill_chunked writing y = RMSNorm(o) * norm_weight * SiLU(z) per
    (token, V head) row instead of o.  z: [T, hv, dv] (a view with a free row
    stride); norm_weight [dv] fp32.  Returns y [T, hv, dv].  workspace as for
    gdn_prefill_chunked."""
    _cuda(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices, final_state_indices,
          z, norm_weight)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    zs = _heads_view(z, hv, dv, "z")
    _need(q.dtype == k.dtype == v.dtype == z.dtype, "q, k, v, z: one dtype")
    _need(z.shape[0] == T, "z: [T, hv, dv]")
    _need(norm_weight.dtype == torch.float32 and norm_weight.is_contiguous()
          and norm_weight.shape == (dv,), "norm_weight: [dv] fp32")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32 and g.is_contiguous()
          and beta.is_contiguous() and g.shape == (T, hv) and beta.shape == (T, hv), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    _i32_vec(cu_seqlens, "cu_seqlens")
    n = cu_seqlens.numel() - 1
    for name, t in (("initial_state_indices", initial_state_indices),
                    ("final_state_indices", final_state_indices)):
        if t is not None:
            _i32_vec(t, name)
            _need(t.numel() == n, f"{name}: [n_seqs]")
    y = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if y is None else y
    _need(y.is_contiguous() and y.shape == (T, hv, dv), "y: [T, hv, dv] contiguous")
    dt = _dtype_code(q)
    if workspace is False:
        workspace = None
    elif workspace is None:
        need = gdn_prefill_workspace_size(n, T, hv, dk, dv, chunk, dt)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    else:
        _cuda(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_prefill_chunked_gated(
        _ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g), _ptr(beta), _ptr(cu_seqlens), n, T, hqk,
        hv, dk, dv, float(scale), int(l2norm_qk), chunk, _ptr(state_pool), state_pool.shape[0],
        _ptr(initial_state_indices), _ptr(final_state_indices), _ptr(z), zs, _ptr(norm_weight),
        float(norm_eps), _ptr(y), dt, _ptr(workspace), wbytes, _stream(q.device)),
        "gdn_prefill_chunked_gated")
    return y


def gdn_mixed_batch(q, k, v, g, beta, cu_seqlens, n_decode, state_pool, initial_state_indices,
                    final_state_indices, scale, decode_in_place=True, chunk=64, l2norm_qk=True,
                    o=None, workspace=None):
    """A serving step's mixed batch: sequences 0 .. n_decode-1 are one-token
    decode rows (rows 0 .. n_decode-1) continuing the states in
    initial_state_indices (in place, or into final_state_indices when
    decode_in_place is False); the rest go through the chunked prefill with
    both index arrays.  Shapes as gdn_prefill_chunked; workspace as there,
    sized for the prefill sequences."""
    _cuda(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices, final_state_indices)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v: one dtype")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32 and g.is_contiguous()
          and beta.is_contiguous() and g.shape == (T, hv) and beta.shape == (T, hv), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    _i32_vec(cu_seqlens, "cu_seqlens")
    n = cu_seqlens.numel() - 1
    _need(0 <= n_decode <= n and n_decode <= T, "n_decode: 0 .. n_seqs")
    for name, t in (("initial_state_indices", initial_state_indices),
                    ("final_state_indices", final_state_indices)):
        if t is not None:
            _i32_vec(t, name)
            _need(t.numel() == n, f"{name}: [n_seqs]")
    o = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if o is None else o
    _need(o.is_contiguous() and o.shape == (T, hv, dv), "o: [T, hv, dv] contiguous")
    dt = _dtype_code(q)
    if workspace is False:
        workspace = None
    elif workspace is None:
        need = gdn_prefill_workspace_size(n - n_decode, T, hv, dk, dv, chunk, dt) if n > n_decode else 0
        # + 512 bytes: room for the work counter of the decode beside the prefill
        workspace = torch.empty(need + 512, dtype=torch.uint8, device=q.device) if need else None
    else:
        _cuda(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_mixed_batch(_ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g), _ptr(beta),
                                _ptr(cu_seqlens), n, int(n_decode), T, hqk, hv, dk, dv,
                                float(scale), int(l2norm_qk), chunk, _ptr(state_pool),
                                state_pool.shape[0], _ptr(initial_state_indices),
                                _ptr(final_state_indices), int(bool(decode_in_place)), _ptr(o),
                                dt, _ptr(workspace), wbytes, _stream(q.device)),
           "gdn_mixed_batch")
    return o


def gdn_prefill_chunked_static(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices,
                               final_state_indices, scale, l2norm_qk=True, o=None):
    """gdn_prefill_chunked for bf16, dk = dv = 128, chunk 64, with the
    library's fixed device scratch instead of a workspace: no allocation in
    the library (o is allocated here unless given).  Raises GdnError
    (GDN_ERR_TOO_LARGE) past PREFILL_STATIC_SCRATCH_BYTES of scratch."""
    _cuda(q, k, v, g, beta, cu_seqlens, state_pool, initial_state_indices, final_state_indices)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    _need(q.dtype == k.dtype == v.dtype == torch.bfloat16 and dk == dv == 128,
          "q, k, v: bf16, head dim 128")
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    _need(g.dtype == torch.float32 and beta.dtype == torch.float32 and g.is_contiguous()
          and beta.is_contiguous() and g.shape == (T, hv) and beta.shape == (T, hv), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    _i32_vec(cu_seqlens, "cu_seqlens")
    n = cu_seqlens.numel() - 1
    for name, t in (("initial_state_indices", initial_state_indices),
                    ("final_state_indices", final_state_indices)):
        if t is not None:
            _i32_vec(t, name)
            _need(t.numel() == n, f"{name}: [n_seqs]")
    o = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if o is None else o
    _need(o.is_contiguous() and o.shape == (T, hv, dv), "o: [T, hv, dv] contiguous")
    _check(_lib.gdn_prefill_chunked_static(_ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g),
                                           _ptr(beta), _ptr(cu_seqlens), n, T, hqk, hv,
                                           float(scale), int(l2norm_qk), _ptr(state_pool),
                                           state_pool.shape[0], _ptr(initial_state_indices),
                                           _ptr(final_state_indices), _ptr(o),
                                           _stream(q.device)),
           "gdn_prefill_chunked_static")
    return o


def gdn_decode_recurrent(q, k, v, g, beta, tokens_per_seq, state_pool, state_indices,
                         snap_indices=None, scale=None, l2norm_qk=True, o=None):
    """Recurrent decode / MTP decode.  q, k [N*tps, hqk, dk]; v [N*tps, hv, dv];
    g, beta [N*tps, hv] fp32; returns o [N*tps, hv, dv]."""
    _cuda(q, k, v, g, beta, state_pool, state_indices, snap_indices)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v: one dtype")
    _i32_vec(state_indices, "state_indices")
    _i32_vec(snap_indices, "snap_indices")
    N = state_indices.numel()
    _need(T == N * tokens_per_seq, "rows != n_seqs * tokens_per_seq")
    _need(g.shape == (T, hv) and beta.shape == (T, hv) and g.dtype == torch.float32
          and beta.dtype == torch.float32 and g.is_contiguous() and beta.is_contiguous(), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    if snap_indices is not None:
        _need(snap_indices.numel() == T, "snap_indices: [n_seqs, tps]")
    scale = dk ** -0.5 if scale is None else scale
    o = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if o is None else o
    _check(_lib.gdn_decode_recurrent(_ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g), _ptr(beta), N,
                                     tokens_per_seq, hqk, hv, dk, dv, float(scale), int(l2norm_qk),
                                     _ptr(state_pool), state_pool.shape[0], _ptr(state_indices),
                                     _ptr(snap_indices), _ptr(o), _dtype_code(q),
                                     _stream(q.device)), "gdn_decode_recurrent")
    return o


def gdn_decode_recurrent_gated(q, k, v, g, beta, tokens_per_seq, state_pool, state_indices, z,
                               norm_weight, norm_eps=1e-6, snap_indices=None, scale=None,
                               l2norm_qk=True, y=None):
    """gdn_decode_recurrent with the gated RMSNorm fused into the output:
    returns y = o / sqrt(mean(o^2) + eps) * norm_weight * SiLU(z), [N*tps, hv, dv].
    z: [N*tps, hv, dv] (a view with a free row stride), norm_weight [dv] fp32."""
    _cuda(q, k, v, g, beta, state_pool, state_indices, snap_indices, z, norm_weight)
    T, hqk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    qs = _heads_view(q, hqk, dk, "q")
    ks = _heads_view(k, hqk, dk, "k")
    vs = _heads_view(v, hv, dv, "v")
    zs = _heads_view(z, hv, dv, "z")
    _need(q.dtype == k.dtype == v.dtype == z.dtype, "q, k, v, z: one dtype")
    _need(norm_weight.dtype == torch.float32 and norm_weight.is_contiguous()
          and norm_weight.shape == (dv,), "norm_weight: [dv] fp32")
    _i32_vec(state_indices, "state_indices")
    _i32_vec(snap_indices, "snap_indices")
    N = state_indices.numel()
    _need(T == N * tokens_per_seq and z.shape[0] == T, "rows != n_seqs * tokens_per_seq")
    _need(g.shape == (T, hv) and beta.shape == (T, hv) and g.dtype == torch.float32
          and beta.dtype == torch.float32 and g.is_contiguous() and beta.is_contiguous(), "g, beta")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, dv, dk), "state_pool: [slots, hv, dv, dk] fp32")
    if snap_indices is not None:
        _need(snap_indices.numel() == T, "snap_indices: [n_seqs, tps]")
    scale = dk ** -0.5 if scale is None else scale
    y = torch.empty((T, hv, dv), dtype=q.dtype, device=q.device) if y is None else y
    _need(y.is_contiguous() and y.shape == (T, hv, dv), "y: [T, hv, dv] contiguous")
    _check(_lib.gdn_decode_recurrent_gated(
        _ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(g), _ptr(beta), N, tokens_per_seq, hqk, hv,
        dk, dv, float(scale), int(l2norm_qk), _ptr(state_pool), state_pool.shape[0],
        _ptr(state_indices), _ptr(snap_indices), _ptr(z), zs, _ptr(norm_weight),
        float(norm_eps), _ptr(y), _dtype_code(q), _stream(q.device)), "gdn_decode_recurrent_gated")
    return y


def gdn_decode_step_workspace_size(n_seqs, hqk, hv) -> int:
    return int(_lib.gdn_decode_step_workspace_size(n_seqs, hqk, hv))


def gdn_decode_step_fused(x, conv_weight, conv_state_pool, a, b, A_log, dt_bias, hqk,
                          state_pool, state_indices, scale=None, conv_bias=None, o=None,
                          workspace=None):
    """One decode step: conv update + SiLU of the raw q|k|v stream x [N, C],
    gating from a, b [N, hv], L2 norms and the recurrent update.  Same result
    as causal_conv1d_update + gdn_gating + gdn_decode_recurrent.  bf16,
    dk = dv = 128; both pools use state_indices.  Returns o [N, hv, 128].

    workspace: None allocates the scratch gdn_decode_step_workspace_size asks
    for (the step then runs as the conv / gates kernel and the streaming
    decode behind it); a uint8 CUDA tensor is used as given; False passes
    none, which selects the single fused kernel."""
    _cuda(x, conv_weight, conv_state_pool, a, b, A_log, dt_bias, state_pool, state_indices,
          conv_bias)
    N, C = x.shape
    hv = a.shape[1]
    _need(x.dtype == torch.bfloat16 and x.stride(1) == 1, "x: bf16 rows")
    _need(C == 2 * hqk * 128 + hv * 128, "x: 2*hqk*128 + hv*128 channels")
    _need(conv_weight.shape == (C, 4) and conv_weight.is_contiguous()
          and conv_weight.dtype == torch.bfloat16, "conv_weight: [C, 4] bf16")
    _need(conv_state_pool.dtype == torch.bfloat16 and conv_state_pool.is_contiguous()
          and conv_state_pool.shape[1:] == (3, C), "conv_state_pool: [slots, 3, C] bf16")
    _need(a.shape == (N, hv) and b.shape == (N, hv) and a.is_contiguous() and b.is_contiguous()
          and a.dtype == b.dtype == torch.bfloat16, "a, b: [N, hv] bf16")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, 128, 128), "state_pool: [slots, hv, 128, 128] fp32")
    _need(conv_state_pool.shape[0] == state_pool.shape[0], "pools: same slot count")
    _i32_vec(state_indices, "state_indices")
    _need(state_indices.numel() == N, "state_indices: [N]")
    scale = 128 ** -0.5 if scale is None else scale
    o = torch.empty((N, hv, 128), dtype=torch.bfloat16, device=x.device) if o is None else o
    _need(o.is_contiguous() and o.shape == (N, hv, 128), "o: [N, hv, 128] contiguous")
    if workspace is False:
        workspace = None
    elif workspace is None:
        need = gdn_decode_step_workspace_size(N, hqk, hv)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    else:
        _cuda(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.gdn_decode_step_fused(
        _ptr(x), x.stride(0), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state_pool), _ptr(a),
        _ptr(b), _ptr(A_log), _ptr(dt_bias), N, hqk, hv, float(scale), _ptr(state_pool),
        state_pool.shape[0], _ptr(state_indices), _ptr(workspace), wbytes, _ptr(o),
        _stream(x.device)), "gdn_decode_step_fused")
    return o


def gdn_prefill_layer_workspace_size(n_seqs, n_tokens, hqk, hv) -> int:
    return int(_lib.gdn_prefill_layer_workspace_size(n_seqs, n_tokens, hqk, hv))


def _layer_args(x, conv_weight, conv_state_pool, conv_state_indices, has_initial_state, a, b,
                A_log, dt_bias, cu_seqlens, hqk, state_pool, initial_state_indices,
                final_state_indices, conv_bias, out, workspace):
    """Checks and marshalling shared by the two layer calls: the leading
    arguments up to the index arrays, the output tensor and the workspace."""
    _cuda(x, conv_weight, conv_state_pool, conv_state_indices, a, b, A_log, dt_bias, cu_seqlens,
          state_pool, initial_state_indices, final_state_indices, conv_bias, has_initial_state)
    T, C = x.shape
    hv = a.shape[1]
    _need(x.dtype == torch.bfloat16 and x.stride(1) == 1, "x: bf16 rows")
    _need(C == 2 * hqk * 128 + hv * 128, "x: 2*hqk*128 + hv*128 channels")
    _need(conv_weight.shape == (C, 4) and conv_weight.is_contiguous()
          and conv_weight.dtype == torch.bfloat16, "conv_weight: [C, 4] bf16")
    _need(conv_state_pool.dtype == torch.bfloat16 and conv_state_pool.is_contiguous()
          and conv_state_pool.shape[1:] == (3, C), "conv_state_pool: [slots, 3, C] bf16")
    _need(a.shape == (T, hv) and b.shape == (T, hv) and a.is_contiguous() and b.is_contiguous()
          and a.dtype == b.dtype == torch.bfloat16, "a, b: [T, hv] bf16")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, 128, 128), "state_pool: [slots, hv, 128, 128] fp32")
    _i32_vec(cu_seqlens, "cu_seqlens")
    n = cu_seqlens.numel() - 1
    for name, t in (("conv_state_indices", conv_state_indices),
                    ("initial_state_indices", initial_state_indices),
                    ("final_state_indices", final_state_indices)):
        if t is not None:
            _i32_vec(t, name)
            _need(t.numel() == n, f"{name}: [n_seqs]")
    if has_initial_state is not None:
        _need(has_initial_state.dtype == torch.uint8 and has_initial_state.numel() == n,
              "has_initial_state: [n_seqs] uint8")
    out = torch.empty((T, hv, 128), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out.is_contiguous() and out.shape == (T, hv, 128), "output: [T, hv, 128] contiguous")
    if workspace is None:
        need = gdn_prefill_layer_workspace_size(n, T, hqk, hv)
        workspace = torch.empty(need + 1024, dtype=torch.uint8, device=x.device) if need else None
        if workspace is not None:   # 1 KiB alignment
            off = (-workspace.data_ptr()) % 1024
            workspace = workspace[off:off + need]
    else:
        _cuda(workspace)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lead = (_ptr(x), x.stride(0), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state_pool),
            conv_state_pool.shape[0], _ptr(conv_state_indices), _ptr(has_initial_state), _ptr(a),
            _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(cu_seqlens), n, T, hqk, hv)
    tail = (_ptr(state_pool), state_pool.shape[0], _ptr(initial_state_indices),
            _ptr(final_state_indices))
    return lead, tail, out, (_ptr(workspace), wbytes, _stream(x.device))


def gdn_prefill_layer(x, conv_weight, conv_state_pool, conv_state_indices, has_initial_state, a, b,
                      A_log, dt_bias, cu_seqlens, hqk, state_pool, initial_state_indices,
                      final_state_indices, scale=None, conv_bias=None, o=None, workspace=None):
    """The prefill side of the layer in one call: the causal conv + SiLU of the
    raw q|k|v stream x [T, C] (conv states as causal_conv1d_fwd), then the
    chunked prefill on its q, k, v with the gates formed from the raw a, b
    [T, hv] inside the prefill.  bf16, dk = dv = 128, chunk 64.  Returns o
    [T, hv, 128].  workspace: None allocates gdn_prefill_layer_workspace_size
    bytes; a uint8 CUDA tensor is used as given."""
    lead, tail, o, ws = _layer_args(x, conv_weight, conv_state_pool, conv_state_indices,
                                    has_initial_state, a, b, A_log, dt_bias, cu_seqlens, hqk,
                                    state_pool, initial_state_indices, final_state_indices,
                                    conv_bias, o, workspace)
    scale = 128 ** -0.5 if scale is None else scale
    _check(_lib.gdn_prefill_layer(*lead, float(scale), *tail, _ptr(o), *ws), "gdn_prefill_layer")
    return o


def gdn_prefill_layer_gated(x, conv_weight, conv_state_pool, conv_state_indices, has_initial_state,
                            a, b, A_log, dt_bias, cu_seqlens, hqk, state_pool,
                            initial_state_indices, final_state_indices, z, norm_weight,
                            norm_eps=1e-6, scale=None, conv_bias=None, y=None, workspace=None):
    """gdn_prefill_layer writing the gated RMSNorm y = o / rms(o) * w *
    SiLU(z) per (token, V head) row instead of o; z [T, hv, 128] or
    [T, hv*128] bf16 (row stride free), norm_weight [128] fp32.  Returns y
    [T, hv, 128]."""
    _cuda(z, norm_weight)
    zs = _heads_view(z, a.shape[1], 128, "z")
    _need(z.dtype == torch.bfloat16 and z.shape[0] == x.shape[0], "z: [T, hv, 128] bf16")
    _need(norm_weight.dtype == torch.float32 and norm_weight.is_contiguous()
          and norm_weight.numel() == 128, "norm_weight: [128] fp32")
    lead, tail, y, ws = _layer_args(x, conv_weight, conv_state_pool, conv_state_indices,
                                    has_initial_state, a, b, A_log, dt_bias, cu_seqlens, hqk,
                                    state_pool, initial_state_indices, final_state_indices,
                                    conv_bias, y, workspace)
    scale = 128 ** -0.5 if scale is None else scale
    _check(_lib.gdn_prefill_layer_gated(*lead, float(scale), *tail, _ptr(z), zs,
                                        _ptr(norm_weight), float(norm_eps), _ptr(y), *ws),
           "gdn_prefill_layer_gated")
    return y


def gdn_mtp_step_fused(x, tokens_per_seq, conv_weight, conv_state_pool, a, b, A_log, dt_bias,
                       hqk, state_pool, state_indices, snap_indices, scale=None, conv_bias=None,
                       o=None):
    """One MTP draft step in one kernel: conv update + SiLU of the raw q|k|v
    stream x [N * tps, C] (row i * tps + t), gating from a, b [N * tps, hv],
    L2 norms and the recurrent update over the tps tokens, with the conv and
    recurrent states after token t written to slot snap_indices[i][t] of
    both pools (the source slots are only read).  Returns o [N * tps, hv, 128]."""
    _cuda(x, conv_weight, conv_state_pool, a, b, A_log, dt_bias, state_pool, state_indices,
          snap_indices, conv_bias)
    T, C = x.shape
    hv = a.shape[1]
    _i32_vec(state_indices, "state_indices")
    _i32_vec(snap_indices, "snap_indices")
    N = state_indices.numel()
    _need(T == N * tokens_per_seq, "x rows != n_seqs * tokens_per_seq")
    _need(snap_indices.numel() == T, "snap_indices: [n_seqs, tps]")
    _need(x.dtype == torch.bfloat16 and x.stride(1) == 1, "x: bf16 rows")
    _need(C == 2 * hqk * 128 + hv * 128, "x: 2*hqk*128 + hv*128 channels")
    _need(conv_weight.shape == (C, 4) and conv_weight.is_contiguous()
          and conv_weight.dtype == torch.bfloat16, "conv_weight: [C, 4] bf16")
    _need(conv_state_pool.dtype == torch.bfloat16 and conv_state_pool.is_contiguous()
          and conv_state_pool.shape[1:] == (3, C), "conv_state_pool: [slots, 3, C] bf16")
    _need(a.shape == (T, hv) and b.shape == (T, hv) and a.is_contiguous() and b.is_contiguous()
          and a.dtype == b.dtype == torch.bfloat16, "a, b: [N*tps, hv] bf16")
    _need(state_pool.dtype == torch.float32 and state_pool.is_contiguous()
          and state_pool.shape[1:] == (hv, 128, 128), "state_pool: [slots, hv, 128, 128] fp32")
    _need(conv_state_pool.shape[0] == state_pool.shape[0], "pools: same slot count")
    scale = 128 ** -0.5 if scale is None else scale
    o = torch.empty((T, hv, 128), dtype=torch.bfloat16, device=x.device) if o is None else o
    _need(o.is_contiguous() and o.shape == (T, hv, 128), "o: [N*tps, hv, 128] contiguous")
    _check(_lib.gdn_mtp_step_fused(
        _ptr(x), x.stride(0), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state_pool), _ptr(a),
        _ptr(b), _ptr(A_log), _ptr(dt_bias), N, tokens_per_seq, hqk, hv, float(scale),
        _ptr(state_pool), state_pool.shape[0], _ptr(state_indices), _ptr(snap_indices), _ptr(o),
        _stream(x.device)), "gdn_mtp_step_fused")
    return o


def gdn_gated_rmsnorm(o, z, weight, eps=1e-6, y=None):
    """y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z) per (token, head) row.
    o [T, hv, dv] contiguous; z [T, hv, dv] (a view with a free row stride);
    weight [dv] fp32.  y defaults to a new tensor; pass y=o for in place."""
    _cuda(o, z, weight)
    T, hv, dv = o.shape
    _need(o.is_contiguous(), "o: contiguous")
    zs = _heads_view(z, hv, dv, "z")
    _need(z.shape == o.shape and z.dtype == o.dtype, "z: same shape and dtype as o")
    _need(weight.dtype == torch.float32 and weight.is_contiguous() and weight.shape == (dv,),
          "weight: [dv] fp32")
    y = torch.empty_like(o) if y is None else y
    _need(y.is_contiguous() and y.shape == o.shape and y.dtype == o.dtype, "y: like o")
    _check(_lib.gdn_gated_rmsnorm(_ptr(o), _ptr(z), zs, _ptr(weight), T, hv, dv, float(eps),
                                  _ptr(y), _dtype_code(o), _stream(o.device)), "gdn_gated_rmsnorm")
    return y


def gdn_state_snapshot(pool, src, dst):
    """pool[dst[i]] <- pool[src[i]] for whole slots (any pool dtype)."""
    _cuda(pool, src, dst)
    _i32_vec(src, "src")
    _i32_vec(dst, "dst")
    _need(src.numel() == dst.numel(), "src/dst length")
    _need(pool.is_contiguous(), "pool must be contiguous")
    slot_bytes = pool[0].numel() * pool.element_size()
    _check(_lib.gdn_state_snapshot(_ptr(pool), pool.shape[0], slot_bytes, _ptr(src), _ptr(dst),
                                   src.numel(), _stream(pool.device)), "gdn_state_snapshot")


def gdn_get_device_status(clear=True, device=None) -> int:
    """Device status word (DEVSTAT_* bits); synchronises the current stream."""
    out = ctypes.c_uint32(0)
    _check(_lib.gdn_get_device_status(ctypes.byref(out), int(clear), _stream(device)),
           "gdn_get_device_status")
    return int(out.value)


def gdn_debug_set_wait_limit(limit_ns=0, drop_prep_loads=False, device=None):
    """Test control of the two-kernel prefill's failure path: the limit of its
    bounded waits (0 = the default, one second) and whether the prep kernel
    skips its K|Q loads (its waits then run out and the call sets
    DEVSTAT_TIMEOUT; its results are undefined).  Synchronises the stream."""
    _check(_lib.gdn_debug_set_wait_limit(int(limit_ns), int(bool(drop_prep_loads)),
                                         _stream(device)), "gdn_debug_set_wait_limit")
