"""GB300 (sm_103a) chunked gated delta rule forward scan.

A thin ctypes binding over libgdn.so (include/gdn.h). PyTorch supplies
device memory and the current stream; every step of the computation runs in
the library's CUDA kernels. There is no CPU fallback: if the library is not
built, or no GPU is present, calls fail loudly.

Entry points mirror the C ABI:
  gdn_prep, gdn_chunk_fwd, gdn_merge, gdn_workspace_size, gdn_status_string,
  gdn_last_device_error, and gdn_forward (prep + one or both scan directions,
  optionally merged).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

__all__ = ["GDNError", "gdn_prep", "gdn_chunk_fwd", "gdn_chunk_fwd_noalloc",
           "gdn_merge", "gdn_frame_fwd", "gdn_frame_workspace_size", "gdn_workspace_size",
           "gdn_status_string", "gdn_last_device_error", "gdn_noalloc_last_device_error",
           "gdn_set_stall_test", "gdn_set_fused", "gdn_forward", "lib",
           "PREP_L2", "PREP_RMS", "PREP_RELU", "gdn_prep_bwd", "gdn_frame_bwd", "gdn_merge_bwd", "profile_enable", "profile_collect", "gdn_set_state_tile",
           "launch_count", "kernel_names"]

F32, BF16 = 0, 1
PREP_L2, PREP_RMS, PREP_RELU = 0x0, 0x1, 0x10
ACCUMULATE, QK_L2NORM = 0x1, 0x2
_STATUS = {0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_DTYPE",
           4: "GDN_ERR_LAYOUT", 5: "GDN_ERR_UNSUPPORTED", 6: "GDN_ERR_CUDA",
           7: "GDN_ERR_TIMEOUT", 8: "GDN_ERR_WORKSPACE", 9: "GDN_ERR_DEVICE"}


class TensorDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("stride_b", ctypes.c_int64), ("stride_t", ctypes.c_int64),
                ("stride_h", ctypes.c_int64)]


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = _STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({gdn_status_string(status)})")


_lib = None


def lib():
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"libgdn.so is not built ({LIB}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB)
    P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_status_string.argtypes = [I]
    L.gdn_workspace_size.restype = ctypes.c_size_t
    L.gdn_workspace_size.argtypes = [I] * 9
    L.gdn_prep.restype = I
    L.gdn_prep.argtypes = [P, TensorDesc, P, TensorDesc, I, I, I, I, I, F, F, P, P]
    L.gdn_chunk_fwd.restype = I
    L.gdn_chunk_fwd.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, P, I, P,
                                TensorDesc, P, P, I, I, I, I, I, I, I, I, P,
                                ctypes.c_size_t, P]
    L.gdn_chunk_fwd_noalloc.restype = I
    L.gdn_chunk_fwd_noalloc.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, P, I, P,
                                        TensorDesc, P, P, I, I, I, I, I, I, I, I, P]
    L.gdn_frame_workspace_size.restype = ctypes.c_size_t
    L.gdn_frame_workspace_size.argtypes = [I] * 7
    L.gdn_frame_fwd.restype = I
    L.gdn_frame_fwd.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, TensorDesc, P, P,
                                I, I, I, I, I, I, I, I, P, ctypes.c_size_t, P]
    L.gdn_seg_workspace_size.restype = ctypes.c_size_t
    L.gdn_seg_workspace_size.argtypes = [I] * 7
    L.gdn_chunk_fwd_seg.restype = I
    L.gdn_chunk_fwd_seg.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, P, TensorDesc, P,
                                    P, I, I, I, I, I, I, I, I, I, P, ctypes.c_size_t, P]
    L.gdn_seg_choose.restype = I
    L.gdn_seg_choose.argtypes = [I] * 7
    L.gdn_state_summary.restype = I
    L.gdn_state_summary.argtypes = [P, TensorDesc, P, TensorDesc, P, P, P, P, P, I, I, I, I, I, I,
                                    I, I, P, ctypes.c_size_t, P]
    L.gdn_bwd_workspace_size.restype = ctypes.c_size_t
    L.gdn_bwd_workspace_size.argtypes = [I] * 9
    L.gdn_bwd_f32_workspace_size.restype = ctypes.c_size_t
    L.gdn_bwd_f32_workspace_size.argtypes = [I] * 9
    L.gdn_chunk_bwd.restype = I
    L.gdn_chunk_bwd.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, P, I, P, TensorDesc,
                                P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, ctypes.c_size_t, P]
    L.gdn_merge_bwd.restype = I
    L.gdn_merge_bwd.argtypes = [P, TensorDesc, P, P, TensorDesc, P, P, P, P, I, I, I, I,
                                ctypes.c_float, P]
    L.gdn_prep_bwd.restype = I
    L.gdn_prep_bwd.argtypes = [P, TensorDesc, P, P, I, I, I, I, I, ctypes.c_float, ctypes.c_float, P]
    L.gdn_frame_bwd_workspace_size.restype = ctypes.c_size_t
    L.gdn_frame_bwd_workspace_size.argtypes = [I] * 7
    L.gdn_frame_bwd.restype = I
    L.gdn_frame_bwd.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, TensorDesc, P, P, P, P,
                                P, P, P, P, I, I, I, I, I, I, I, I, P, ctypes.c_size_t, P]
    L.gdn_bidir_workspace_size.restype = ctypes.c_size_t
    L.gdn_bidir_workspace_size.argtypes = [I] * 9
    L.gdn_chunk_fwd_bidir.restype = I
    L.gdn_chunk_fwd_bidir.argtypes = [P, P, TensorDesc, P, TensorDesc, P, P, P, P, P, P, I, P,
                                      TensorDesc, P, I, I, I, I, I, I, I, P, ctypes.c_size_t, P]
    L.gdn_merge.restype = I
    L.gdn_merge.argtypes = [P, TensorDesc, P, P, TensorDesc, P, TensorDesc, I, I, I, I, F, P]
    L.gdn_last_device_error.restype = I
    L.gdn_last_device_error.argtypes = [P, P, ctypes.POINTER(I)]
    L.gdn_noalloc_last_device_error.restype = I
    L.gdn_noalloc_last_device_error.argtypes = [P, ctypes.POINTER(I)]
    L.gdn_set_stall_test.restype = None
    L.gdn_set_stall_test.argtypes = [I, I]
    L.gdn_set_fused.restype = None
    L.gdn_set_fused.argtypes = [I]
    L.gdn_kernel_kinds.restype = I
    L.gdn_kernel_kinds.argtypes = []
    L.gdn_kernel_name.restype = ctypes.c_char_p
    L.gdn_kernel_name.argtypes = [I]
    L.gdn_profile_enable.restype = None
    L.gdn_profile_enable.argtypes = [I]
    L.gdn_set_state_tile.restype = None
    L.gdn_set_state_tile.argtypes = [I]
    L.gdn_profile_collect.restype = I
    L.gdn_profile_collect.argtypes = [ctypes.POINTER(F), ctypes.POINTER(I), I]
    L.gdn_launch_count.restype = ctypes.c_longlong
    L.gdn_launch_count.argtypes = []
    _lib = L
    return L


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise GDNError(3, f"unsupported dtype {t.dtype}")


def _desc(t) -> TensorDesc:
    """Descriptor of a 4-D (B, T, H, D) view with a contiguous last dim."""
    if t.dim() != 4:
        raise GDNError(2, f"expected a 4-D (B, T, H, D) tensor, got shape {tuple(t.shape)}")
    if t.stride(3) != 1:
        raise GDNError(4, "the last dimension must be contiguous")
    return TensorDesc(_dtype_code(t), 0, t.stride(0), t.stride(1), t.stride(2))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _state_shape(n_seq, H, K, V, den, **states):
    """State tensors are (n_seq, H, K, V), with the denominator's z column
    (V + 1) when den is given; the library cannot see a buffer's size."""
    want = (n_seq, H, K, V + (1 if den is not None else 0))
    for name, t in states.items():
        if t is not None and tuple(t.shape) != want:
            raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")


def _f32(t, name):
    torch = _torch()
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise GDNError(3 if t.dtype != torch.float32 else 4,
                       f"{name} must be a contiguous float32 tensor")
    return t


def gdn_workspace_size(B, T, H, K, V, n_seq, varlen, dtype, with_den) -> int:
    return int(lib().gdn_workspace_size(B, T, H, K, V, n_seq, int(bool(varlen)),
                                        dtype, int(bool(with_den))))


def gdn_prep(x, y=None, mode=PREP_L2, scale=1.0, eps=1e-6, inv_rms=None, stream=None):
    """q/k preparation on the GPU (see include/gdn.h). x: (B, T, H, D).
    Returns y (allocated like x when not given)."""
    torch = _torch()
    B, T, H, D = x.shape
    if y is None:
        y = torch.empty((B, T, H, D), dtype=x.dtype, device=x.device)
    if inv_rms is not None:
        _f32(inv_rms, "inv_rms")
    st = lib().gdn_prep(_ptr(x), _desc(x), _ptr(y), _desc(y), B, T, H, D, int(mode),
                        float(scale), float(eps), _ptr(inv_rms), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_prep")
    return y


def gdn_chunk_fwd(q, k, v, beta, g=None, gk=None, h0=None, cu_seqlens=None, out=None,
                  h_final=None, den=None, reverse=False, accumulate=False,
                  qk_l2norm=False, workspace=None, stream=None, out_dtype=None):
    """One direction of the chunked scan (see include/gdn.h).

    q, k: (B, T, H, K); v: (B, T, H, V); beta, g: (B, T, H) fp32;
    gk: (B, T, H, K) fp32; h0/h_final: (n_seq, H, K, V) fp32, or
    (n_seq, H, K, V + 1) with `den` (column V: the denominator's z state);
    cu_seqlens: int32 device tensor (n_seq + 1) with B == 1;
    den: (B, H, T) fp32. Missing `out` / `workspace` are allocated with
    torch. Returns out."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    n_seq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous()):
        raise GDNError(3, "cu_seqlens must be a contiguous int32 tensor")
    for name, t in (("beta", beta), ("g", g), ("gk", gk), ("h0", h0), ("h_final", h_final),
                    ("den", den)):
        _f32(t, name)
    _state_shape(n_seq, H, K, V, den, h0=h0, h_final=h_final)
    if out is None:
        out = torch.empty((B, T, H, V), dtype=out_dtype or q.dtype, device=q.device)
    dt = _dtype_code(q)
    need = gdn_workspace_size(B, T, H, K, V, n_seq, cu_seqlens is not None, dt, den is not None)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    flags = (ACCUMULATE if accumulate else 0) | (QK_L2NORM if qk_l2norm else 0)
    # an empty den (T = 0) may have no address; any non-NULL pointer tells
    # the library that the state carries the z column (nothing is written)
    den_p = _ptr(workspace) if den is not None and den.numel() == 0 else _ptr(den)
    st = lib().gdn_chunk_fwd(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta),
        _ptr(h0), _ptr(cu_seqlens), n_seq, _ptr(out), _desc(out), _ptr(h_final), den_p,
        B, T, H, K, V, 64, int(bool(reverse)), flags, _ptr(workspace),
        workspace.numel(), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_chunk_fwd")
    return out


def gdn_seg_workspace_size(B, T, H, K, V, with_den, segment_len) -> int:
    return int(lib().gdn_seg_workspace_size(B, T, H, K, V, int(bool(with_den)), int(segment_len)))


def gdn_seg_choose(B, T, H, K, V, with_den, n_sm) -> int:
    """segment_len for gdn_chunk_fwd_seg on a GPU with n_sm SMs (host
    arithmetic in the library; see include/gdn.h)."""
    return int(lib().gdn_seg_choose(B, T, H, K, V, int(bool(with_den)), int(n_sm)))


def gdn_chunk_fwd_seg(q, k, v, beta, segment_len, g=None, gk=None, h0=None, out=None,
                      h_final=None, den=None, reverse=False, accumulate=False,
                      qk_l2norm=False, workspace=None, stream=None, out_dtype=None):
    """gdn_chunk_fwd with segment-parallel state passing (dense bf16
    batches; see include/gdn.h). segment_len: tokens per segment, a multiple
    of 64. Returns out."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    for name, t in (("beta", beta), ("g", g), ("gk", gk), ("h0", h0), ("h_final", h_final),
                    ("den", den)):
        _f32(t, name)
    _state_shape(B, H, K, V, den, h0=h0, h_final=h_final)
    if out is None:
        out = torch.empty((B, T, H, V), dtype=out_dtype or q.dtype, device=q.device)
    need = gdn_seg_workspace_size(B, T, H, K, V, den is not None, segment_len)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    flags = (ACCUMULATE if accumulate else 0) | (QK_L2NORM if qk_l2norm else 0)
    st = lib().gdn_chunk_fwd_seg(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta),
        _ptr(h0), _ptr(out), _desc(out), _ptr(h_final), _ptr(den), B, T, H, K, V, 64,
        int(bool(reverse)), flags, int(segment_len), _ptr(workspace), workspace.numel(),
        _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_chunk_fwd_seg")
    return out


def gdn_state_summary(k, v, beta, segment_len, g=None, gk=None, with_transition=True,
                      qk_l2norm=False, workspace=None, stream=None):
    """Per-segment affine summaries (see include/gdn.h): returns
    (state_ext (n_seg, B, H, K, V), transition (n_seg, B, H, K, K) or None),
    fp32, with h_out = transition @ h_in + state_ext per segment."""
    torch = _torch()
    B, T, H, K = k.shape
    V = v.shape[3]
    for name, t in (("beta", beta), ("g", g), ("gk", gk)):
        _f32(t, name)
    n_seg = -(-T // int(segment_len)) if segment_len > 0 else 0
    ext = torch.empty((n_seg, B, H, K, V), dtype=torch.float32, device=k.device)
    tr = (torch.empty((n_seg, B, H, K, K), dtype=torch.float32, device=k.device)
          if with_transition else None)
    need = gdn_workspace_size(B, T, H, K, V, B, 0, BF16, 0)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=k.device)
    st = lib().gdn_state_summary(
        _ptr(k), _desc(k), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta), _ptr(ext), _ptr(tr),
        B, T, H, K, V, 64, int(segment_len), QK_L2NORM if qk_l2norm else 0, _ptr(workspace),
        workspace.numel(), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_state_summary")
    return ext, tr


def gdn_bwd_workspace_size(B, T, H, K, V, n_seq=None, varlen=False, perkey=False,
                           with_den=False, fp32=False) -> int:
    fn = lib().gdn_bwd_f32_workspace_size if fp32 else lib().gdn_bwd_workspace_size
    return int(fn(B, T, H, K, V, B if n_seq is None else n_seq, int(bool(varlen)), int(bool(perkey)),
                  int(bool(with_den))))


def gdn_chunk_bwd(q, k, v, beta, g, dout, h0=None, dh_final=None, reverse=False,
                  qk_l2norm=False, with_dh0=None, workspace=None, stream=None, gk=None,
                  cu_seqlens=None, dden=None):
    """Gradients of one direction of the scan for L = sum(dout * o) +
    sum(dh_final * h_final) (see include/gdn.h). q, k (B, T, H, K), v and
    dout (B, T, H, V), all bf16 (the chunked tensor-core backward) or all
    fp32 (the fp32 token recurrence in reverse); beta, g (B, T, H), h0 / dh_final (n_seq, H, K,
    V) fp32 (V + 1 columns with dden, the denominator's upstream gradient
    (B, H, T)); cu_seqlens: int32 (n_seq + 1) with B == 1. Returns a dict of
    fp32 tensors dq, dk, dv, dbeta, dg and, unless reverse (or
    with_dh0=False), dh0."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    n_seq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous()):
        raise GDNError(3, "cu_seqlens must be a contiguous int32 tensor")
    for name, t in (("beta", beta), ("g", g), ("gk", gk), ("h0", h0), ("dh_final", dh_final),
                    ("dden", dden)):
        _f32(t, name)
    _state_shape(n_seq, H, K, V, dden, h0=h0, dh_final=dh_final)
    f32 = dict(dtype=torch.float32, device=q.device)
    res = {"dq": torch.empty((B, T, H, K), **f32), "dk": torch.empty((B, T, H, K), **f32),
           "dv": torch.empty((B, T, H, V), **f32), "dbeta": torch.empty((B, T, H), **f32),
           "dg": torch.empty((B, T, H) if gk is None else (B, T, H, K), **f32)}
    if with_dh0 is None:
        with_dh0 = not reverse
    if with_dh0:
        res["dh0"] = torch.empty((n_seq, H, K, V + (dden is not None)), **f32)
    need = gdn_bwd_workspace_size(B, T, H, K, V, n_seq, cu_seqlens is not None, gk is not None,
                                  dden is not None, fp32=q.dtype == torch.float32)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().gdn_chunk_bwd(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta), _ptr(h0),
        _ptr(cu_seqlens), n_seq, _ptr(dout), _desc(dout), _ptr(dden), _ptr(dh_final), _ptr(res["dq"]),
        _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["dbeta"]), _ptr(res["dg"]),
        _ptr(res.get("dh0")), B, T, H, K, V, 64, int(bool(reverse)),
        QK_L2NORM if qk_l2norm else 0, _ptr(workspace), workspace.numel(), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_chunk_bwd")
    return res


def gdn_bidir_workspace_size(B, T, H, K, V, n_seq, varlen, dtype, with_den) -> int:
    return int(lib().gdn_bidir_workspace_size(B, T, H, K, V, n_seq, int(bool(varlen)), dtype,
                                              int(bool(with_den))))


def gdn_chunk_fwd_bidir(q, k, v, beta, g=None, gk=None, g_bwd=None, beta_bwd=None,
                        cu_seqlens=None, out=None, den=None, qk_l2norm=False, workspace=None,
                        stream=None):
    """Both directions of the bidirectional scan, run concurrently (see
    include/gdn.h): out = num_fwd + num_bwd, den = den_fwd + den_bwd.
    Returns out (allocated in q's dtype when not given)."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    n_seq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    for name, t in (("beta", beta), ("g", g), ("gk", gk), ("g_bwd", g_bwd),
                    ("beta_bwd", beta_bwd), ("den", den)):
        _f32(t, name)
    if out is None:
        out = torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    need = gdn_bidir_workspace_size(B, T, H, K, V, n_seq, cu_seqlens is not None, _dtype_code(q),
                                    den is not None)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().gdn_chunk_fwd_bidir(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta), _ptr(g_bwd),
        _ptr(beta_bwd), _ptr(cu_seqlens), n_seq, _ptr(out), _desc(out), _ptr(den), B, T, H, K, V,
        64, QK_L2NORM if qk_l2norm else 0, _ptr(workspace), workspace.numel(), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_chunk_fwd_bidir")
    return out


def gdn_chunk_fwd_noalloc(q, k, v, beta, out, g=None, gk=None, h0=None, cu_seqlens=None,
                          h_final=None, den=None, reverse=False, accumulate=False,
                          qk_l2norm=False, stream=None):
    """gdn_chunk_fwd without a workspace, for callers that cannot allocate
    device memory: the library's built-in scratch buffer is used, and this
    wrapper allocates nothing either (`out`, and h_final / den when wanted,
    must be given). Problems larger than the buffer raise GDN_ERR_WORKSPACE.
    Calls that overlap on the GPU race on the shared buffer."""
    B, T, H, K = q.shape
    V = v.shape[3]
    n_seq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    _state_shape(n_seq, H, K, V, den, h0=h0, h_final=h_final)
    flags = (ACCUMULATE if accumulate else 0) | (QK_L2NORM if qk_l2norm else 0)
    st = lib().gdn_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g), _ptr(gk), _ptr(beta),
        _ptr(h0), _ptr(cu_seqlens), n_seq, _ptr(out), _desc(out), _ptr(h_final), _ptr(den),
        B, T, H, K, V, 64, int(bool(reverse)), flags, _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_chunk_fwd_noalloc")
    return out


def gdn_merge_bwd(num, den, dout, gate=None, eps=1e-6, stream=None):
    """The gradient of gdn_merge (see include/gdn.h) for dout = dL/dout
    (fp32): returns dnum, dden and, with a gate, dgate (fp32)."""
    torch = _torch()
    B, T, H, V = num.shape
    for name, t in (("den", den), ("dout", dout)):
        _f32(t, name)
    f32 = dict(dtype=torch.float32, device=num.device)
    res = {"dnum": torch.empty((B, T, H, V), **f32), "dden": torch.empty((B, H, T), **f32)}
    if gate is not None:
        res["dgate"] = torch.empty((B, T, H, V), **f32)
    gd = _desc(gate) if gate is not None else TensorDesc(_dtype_code(num), 0, 0, 0, 0)
    st = lib().gdn_merge_bwd(_ptr(num), _desc(num), _ptr(den), _ptr(gate), gd, _ptr(dout),
                             _ptr(res["dnum"]), _ptr(res["dden"]), _ptr(res.get("dgate")),
                             B, T, H, V, float(eps), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_merge_bwd")
    return res


def gdn_prep_bwd(x, dy, mode=PREP_L2, scale=1.0, eps=1e-6, dx=None, stream=None):
    """The gradient of gdn_prep (see include/gdn.h): dx = dL/dx for dy =
    dL/dy, x the forward's input (B, T, H, D), dy fp32. Returns dx (fp32)."""
    torch = _torch()
    B, T, H, D = x.shape
    _f32(dy, "dy")
    if dx is None:
        dx = torch.empty((B, T, H, D), dtype=torch.float32, device=x.device)
    st = lib().gdn_prep_bwd(_ptr(x), _desc(x), _ptr(dy), _ptr(dx), B, T, H, D, int(mode),
                            float(scale), float(eps), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_prep_bwd")
    return dx


def gdn_frame_bwd_workspace_size(B, T, H, K, V, frame, with_den) -> int:
    return int(lib().gdn_frame_bwd_workspace_size(B, T, H, K, V, frame, int(bool(with_den))))


def gdn_frame_bwd(q, k, v, beta, g_frame, frame, dout, dden=None, h0=None, dh_final=None,
                  direction=0, with_dh0=None, workspace=None, stream=None):
    """Gradients of the frame-causal rule (see include/gdn.h) for
    L = sum(dout * o) + sum(dden * den) + sum(dh_final * h_final), with
    respect to q and k as gdn_frame_fwd takes them. Returns a dict of fp32
    tensors dq, dk, dv, dbeta, dg_frame and, for direction 0 (unless
    with_dh0=False), dh0 (V + 1 columns with dden)."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    for name, t in (("beta", beta), ("g_frame", g_frame), ("dden", dden), ("h0", h0),
                    ("dh_final", dh_final)):
        _f32(t, name)
    _state_shape(B, H, K, V, dden, h0=h0, dh_final=dh_final)
    f32 = dict(dtype=torch.float32, device=q.device)
    res = {"dq": torch.empty((B, T, H, K), **f32), "dk": torch.empty((B, T, H, K), **f32),
           "dv": torch.empty((B, T, H, V), **f32), "dbeta": torch.empty((B, T, H), **f32),
           "dg_frame": torch.empty((B, T // frame, H), **f32)}
    if with_dh0 is None:
        with_dh0 = direction == 0
    if with_dh0:
        res["dh0"] = torch.empty((B, H, K, V + (dden is not None)), **f32)
    need = gdn_frame_bwd_workspace_size(B, T, H, K, V, frame, dden is not None)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().gdn_frame_bwd(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g_frame), _ptr(beta), _ptr(h0),
        _ptr(dout), _desc(dout), _ptr(dden), _ptr(dh_final), _ptr(res["dq"]), _ptr(res["dk"]),
        _ptr(res["dv"]), _ptr(res["dbeta"]), _ptr(res["dg_frame"]), _ptr(res.get("dh0")),
        B, T, H, K, V, int(frame), int(direction), 0, _ptr(workspace), workspace.numel(),
        _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_frame_bwd")
    return res


def gdn_merge(num, den, gate=None, eps=1e-6, out=None, out_dtype=None, stream=None):
    """out = num / (den + eps) * (silu(gate) if gate is given), see
    include/gdn.h. num, gate: (B, T, H, V); den: (B, H, T) fp32. Returns out
    (allocated when not given: num's dtype, or `out_dtype`)."""
    torch = _torch()
    B, T, H, V = num.shape
    _f32(den, "den")
    if out is None:
        out = torch.empty((B, T, H, V), dtype=out_dtype or num.dtype, device=num.device)
    gd = _desc(gate) if gate is not None else TensorDesc(_dtype_code(num), 0, 0, 0, 0)
    st = lib().gdn_merge(_ptr(num), _desc(num), _ptr(den), _ptr(gate), gd, _ptr(out), _desc(out),
                         B, T, H, V, float(eps), _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_merge")
    return out


def gdn_frame_workspace_size(B, T, H, K, V, frame, with_den) -> int:
    return int(lib().gdn_frame_workspace_size(B, T, H, K, V, frame, int(bool(with_den))))


def gdn_frame_fwd(q, k, v, beta, g_frame, frame, out=None, den=None, h0=None, h_final=None,
                  direction=0, accumulate=False, workspace=None, stream=None, out_dtype=None):
    """The frame-causal form (see include/gdn.h): frames of `frame` tokens
    share the pre-frame state. q, k (B, T, H, K), v (B, T, H, V) bf16 (q, k
    prepared); beta (B, T, H), g_frame (B, T // frame, H) fp32; direction 0
    forward, 1 reverse, 2 both summed; den (B, H, T) fp32. Returns out."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[3]
    for name, t in (("beta", beta), ("g_frame", g_frame), ("h0", h0), ("h_final", h_final),
                    ("den", den)):
        _f32(t, name)
    _state_shape(B, H, K, V, den, h0=h0, h_final=h_final)
    if out is None:
        out = torch.empty((B, T, H, V), dtype=out_dtype or q.dtype, device=q.device)
    need = gdn_frame_workspace_size(B, T, H, K, V, frame, den is not None)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().gdn_frame_fwd(
        _ptr(q), _ptr(k), _desc(q), _ptr(v), _desc(v), _ptr(g_frame), _ptr(beta), _ptr(h0),
        _ptr(out), _desc(out), _ptr(h_final), _ptr(den), B, T, H, K, V, int(frame),
        int(direction), ACCUMULATE if accumulate else 0, _ptr(workspace), workspace.numel(),
        _stream(stream))
    if st != 0:
        raise GDNError(st, "gdn_frame_fwd")
    return out


def gdn_last_device_error(workspace, stream=None) -> int:
    """Synchronise, read and clear the device error word; returns it
    (GDN_DEVERR_* bits: 1 malformed cu_seqlens, 2 a bounded wait gave up)."""
    w = ctypes.c_int(0)
    st = lib().gdn_last_device_error(_ptr(workspace), _stream(stream), ctypes.byref(w))
    if st not in (0, 7, 9):
        raise GDNError(st, "gdn_last_device_error")
    return w.value


def gdn_noalloc_last_device_error(stream=None) -> int:
    """gdn_last_device_error for gdn_chunk_fwd_noalloc's built-in buffer on
    the current device; returns the word."""
    w = ctypes.c_int(0)
    st = lib().gdn_noalloc_last_device_error(_stream(stream), ctypes.byref(w))
    if st not in (0, 7, 9):
        raise GDNError(st, "gdn_noalloc_last_device_error")
    return w.value


def gdn_set_fused(on: bool = True) -> None:
    """Run the bf16 scalar-gate forward as one fused tcgen05 kernel per
    direction (on) or as the split intra-chunk + state passes (off, the
    default); see include/gdn.h."""
    lib().gdn_set_fused(int(bool(on)))


def gdn_set_stall_test(cta: int = -1, limit_us: int = 1000) -> None:
    """Testing aid of the time-out path (see include/gdn.h): block `cta` of
    later intra-chunk and state-pass launches stalls, gives up after about
    limit_us and reports a time-out; cta < 0 turns it off."""
    lib().gdn_set_stall_test(int(cta), int(limit_us))


def gdn_forward(q, k, v, beta, g=None, gk=None, h0=None, cu_seqlens=None,
                prep="l2", bidirectional=False, with_final_state=False, workspace=None,
                stream=None, backward=None, merge=False, gate=None, eps=1e-6, frame=1,
                g_frame=None, segment_len=None):
    """The whole forward: q/k prep, then the causal scan, or the causal plus
    the reverse scan summed with the denominator (bidirectional).

    prep: "l2" (per-(token, head) L2 norm fused into the scan), "rms_relu"
    (full-channel RMSNorm, ReLU, and k scaled by K^-0.5, via gdn_prep), or
    None (q, k used as given).
    backward: optional dict of inputs the reverse direction uses instead of
    the forward ones ("q", "k", "v", "beta", "g", "gk"), e.g. the
    chunk-causal form's gates with -inf at chunk boundaries (the SANA
    `fused_gdn.py` page's decay_bwd / beta_bwd / qkv_bwd).
    merge: also return "merged" = out / (den + eps) * silu(gate) (gdn_merge).
    frame > 1: the frame-causal form (gdn_frame_fwd) with per-frame log
    decays g_frame (B, T // frame, H) in place of g.
    segment_len: segment-parallel state passing (gdn_chunk_fwd_seg; dense
    bf16 inputs) with segments of this many tokens, or "auto" for
    gdn_seg_choose's pick on this device.
    h0 / with_final_state: the causal direction's state in and out,
    (n_seq, H, K, V); bidirectional, (n_seq, H, K, V + 1) with the
    denominator's z state in column V (the reverse direction starts from
    zero at the end of the call, as on the pages).
    Returns a dict with "out" and, as requested, "h_final" / "den" /
    "merged" / "q_inv_rms" / "k_inv_rms"."""
    torch = _torch()
    B, T, H, K = q.shape
    n_seq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    res = {}
    fuse = prep == "l2"
    bw = dict(backward or {})
    unknown = set(bw) - {"q", "k", "v", "beta", "g", "gk"}
    if unknown:
        raise ValueError(f"unknown backward inputs {sorted(unknown)}")
    if (backward or merge) and not bidirectional:
        raise ValueError("backward inputs and merge need bidirectional=True")
    if prep == "rms_relu":
        res["q_inv_rms"] = torch.empty((B, T), dtype=torch.float32, device=q.device)
        res["k_inv_rms"] = torch.empty((B, T), dtype=torch.float32, device=q.device)
        q = gdn_prep(q, mode=PREP_RMS | PREP_RELU, scale=1.0, eps=1e-5,
                     inv_rms=res["q_inv_rms"], stream=stream)
        k = gdn_prep(k, mode=PREP_RMS | PREP_RELU, scale=K ** -0.5, eps=1e-5,
                     inv_rms=res["k_inv_rms"], stream=stream)
        for name, scale in (("q", 1.0), ("k", K ** -0.5)):
            if name in bw:
                bw[name] = gdn_prep(bw[name], mode=PREP_RMS | PREP_RELU, scale=scale, eps=1e-5,
                                    stream=stream)
    elif prep not in ("l2", None):
        raise ValueError(f"unknown prep {prep!r}")
    if frame > 1:
        if backward or merge or gk is not None or cu_seqlens is not None:
            raise ValueError("the frame-causal form takes no backward inputs, merge, gk or varlen")
        if fuse:
            q, k = gdn_prep(q, mode=PREP_L2, stream=stream), gdn_prep(k, mode=PREP_L2, stream=stream)
        if not bidirectional:
            hf = (torch.empty((B, H, K, v.shape[3]), dtype=torch.float32, device=q.device)
                  if with_final_state else None)
            res["out"] = gdn_frame_fwd(q, k, v, beta, g_frame, frame, h0=h0, h_final=hf,
                                       workspace=workspace, stream=stream)
            if hf is not None:
                res["h_final"] = hf
            return res
        if h0 is not None or with_final_state:
            raise ValueError("the bidirectional frame-causal form carries no state")
        den = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
        res["out"] = gdn_frame_fwd(q, k, v, beta, g_frame, frame, den=den, direction=2,
                                   workspace=workspace, stream=stream)
        res["den"] = den
        return res
    if segment_len is not None:
        if cu_seqlens is not None or q.dtype != torch.bfloat16:
            raise ValueError("segment-parallel state passing takes dense bf16 inputs")
        if segment_len == "auto":
            n_sm = torch.cuda.get_device_properties(q.device).multi_processor_count
            segment_len = gdn_seg_choose(B, T, H, K, v.shape[3], bidirectional, n_sm)

    def scan(q, k, v, beta, g, gk, **kw):
        if segment_len:
            return gdn_chunk_fwd_seg(q, k, v, beta, segment_len, g=g, gk=gk, qk_l2norm=fuse,
                                     workspace=workspace, stream=stream, **kw)
        return gdn_chunk_fwd(q, k, v, beta, g=g, gk=gk, cu_seqlens=cu_seqlens, qk_l2norm=fuse,
                             workspace=workspace, stream=stream, **kw)

    if not bidirectional:
        hf = (torch.empty((n_seq, H, K, v.shape[3]), dtype=torch.float32, device=q.device)
              if with_final_state else None)
        res["out"] = scan(q, k, v, beta, g, gk, h0=h0, h_final=hf)
        if hf is not None:
            res["h_final"] = hf
        return res
    den = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    hf = (torch.empty((n_seq, H, K, v.shape[3] + 1), dtype=torch.float32, device=q.device)
          if with_final_state else None)
    if (h0 is None and hf is None and not segment_len and not ({"q", "k", "v", "gk"} & set(bw))
            and not (gk is not None and "g" in bw)):
        # both directions at once, the reverse on the library's second stream
        out = gdn_chunk_fwd_bidir(q, k, v, beta, g=g, gk=gk, g_bwd=bw.get("g"),
                                  beta_bwd=bw.get("beta"), cu_seqlens=cu_seqlens, den=den,
                                  qk_l2norm=fuse, stream=stream,
                                  workspace=workspace if workspace is not None and workspace.numel()
                                  >= gdn_bidir_workspace_size(B, T, H, K, v.shape[3], n_seq,
                                                              cu_seqlens is not None,
                                                              _dtype_code(q), True) else None)
    else:
        out = scan(q, k, v, beta, g, gk, den=den, h0=h0, h_final=hf)
        scan(bw.get("q", q), bw.get("k", k), bw.get("v", v), bw.get("beta", beta), bw.get("g", g),
             bw.get("gk", gk), den=den, out=out, reverse=True, accumulate=True)
    res["out"], res["den"] = out, den
    if hf is not None:
        res["h_final"] = hf
    if merge:
        res["merged"] = gdn_merge(out, den, gate=gate, eps=eps, stream=stream)
    return res


def kernel_names() -> list[str]:
    L = lib()
    return [L.gdn_kernel_name(i).decode() for i in range(L.gdn_kernel_kinds())]


def gdn_set_state_tile(bv: int = 0) -> None:
    """Value columns per state-pass CTA: 0 by the grid, 64 or 128 forced
    (see include/gdn.h)."""
    lib().gdn_set_state_tile(int(bv))


def profile_enable(on: bool = True) -> None:
    lib().gdn_profile_enable(int(bool(on)))


def profile_collect() -> dict:
    """{kernel name: (total device ms, launches)} since the last collect."""
    L = lib()
    n = L.gdn_kernel_kinds()
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    st = L.gdn_profile_collect(ms, cnt, n)
    if st != 0:
        raise GDNError(st, "gdn_profile_collect")
    names = kernel_names()
    return {names[i]: (float(ms[i]), int(cnt[i])) for i in range(n) if cnt[i]}


def launch_count() -> int:
    return int(lib().gdn_launch_count())
