"""GB300-native split-K BF16 decode GEMM: ``C[M, N] = B[M, K] @ A[N, K]^T``.

A thin ctypes binding over the C ABI in ``include/splitk.h``
(``_lib/libsplitk_sm103a.so``, built in-tree by ``__graft_entry__.build()`` or
``split_bf16_gemm_swapped_gb300._build.build_all()``).  It only marshals
arguments: every step of the GEMM runs in the library's sm_103a kernels, and
there is no CPU or PyTorch fallback -- if the library is missing, importing a
function that needs it raises.

PyTorch supplies device memory and streams.  Tensors:
  a  weights      [L, N, K] (or [N, K]) bfloat16, CUDA, contiguous
  b  activations  [L, M, K] (or [M, K]) bfloat16, CUDA, contiguous
  c  output       [L, M, N] (or [M, N]) bfloat16, CUDA, contiguous
"""
from __future__ import annotations

import ctypes
from pathlib import Path

from . import _build

__all__ = [
    "SplitKError", "Plan", "Fault", "library_path", "load_library",
    "splitk_plan", "splitk_plan_for", "splitk_gemm_bf16", "splitk_gemm_bf16_planned",
    "splitk_gemm_bf16_hostio", "splitk_gemm_bf16_zerocopy", "splitk_gemm_bf16_noalloc",
    "splitk_gemm_bf16_bias",
    "splitk_plan_check_for", "splitk_plan_candidates_for", "splitk_tune",
    "splitk_plan_w4a16", "splitk_plan_w4a16_for", "splitk_gemm_w4a16", "splitk_gemm_w4a16_planned",
    "splitk_plan_w8a16", "splitk_plan_w8a16_for", "splitk_gemm_w8a16", "splitk_gemm_w8a16_planned",
    "splitk_get_fault",
    "splitk_get_status",
    "splitk_set_wait_limit_ns", "splitk_debug_inject", "splitk_release", "splitk_cache_info",
    "splitk_strerror", "splitk_version", "splitk_set_trace", "FLAG_NO_PDL",
    "INJECT_SKIP_PUBLISH", "TRACE_SLOTS", "TRACE_FIELDS",
    "STATUS",
]

FLAG_NO_PDL = 0x1
INJECT_SKIP_PUBLISH = 0x1

STATUS = {
    0: "SPLITK_OK", -1: "SPLITK_ERR_INVALID_SHAPE", -2: "SPLITK_ERR_MISALIGNED",
    -3: "SPLITK_ERR_UNSUPPORTED_SPLIT", -4: "SPLITK_ERR_NO_FIT", -5: "SPLITK_ERR_CUDA",
    -6: "SPLITK_ERR_TIMEOUT", -7: "SPLITK_ERR_NULL", -8: "SPLITK_ERR_CACHE_FULL",
    -9: "SPLITK_ERR_UNSUPPORTED_DEVICE", -10: "SPLITK_ERR_BAD_PLAN",
    -11: "SPLITK_ERR_SCRATCH", -12: "SPLITK_ERR_NOT_MAPPED", -13: "SPLITK_ERR_CAPTURE",
}


class SplitKError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        self.name = STATUS.get(self.code, str(code))
        msg = f"{self.name}: {splitk_strerror(self.code)}"
        super().__init__(f"{where}: {msg}" if where else msg)


class Plan(ctypes.Structure):
    _fields_ = [
        ("mma_m", ctypes.c_int), ("mma_n", ctypes.c_int), ("stages", ctypes.c_int),
        ("split_k", ctypes.c_int), ("k_tiles_per_cta", ctypes.c_int),
        ("mailbox_dedicated", ctypes.c_int), ("mailbox_quads", ctypes.c_int),
        ("reduce_rounds", ctypes.c_int), ("grid", ctypes.c_uint * 3),
        ("cluster", ctypes.c_uint * 3), ("smem_bytes", ctypes.c_size_t),
        ("ctas_per_sm", ctypes.c_int), ("pdl_trigger", ctypes.c_int),
        ("reduce_scatter", ctypes.c_int), ("b_resident", ctypes.c_int),
        ("a_tmem_tiles", ctypes.c_int), ("tmem_cols", ctypes.c_uint),
        ("mma_issuers", ctypes.c_int), ("b_loader", ctypes.c_int),
        ("l2_prefetch", ctypes.c_int), ("weight_format", ctypes.c_int),
        ("w4_smem_tiles", ctypes.c_int), ("b_stages", ctypes.c_int),
        ("persistent", ctypes.c_int), ("w4_decoders", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["grid"] = list(self.grid)
        d["cluster"] = list(self.cluster)
        return d

    def __repr__(self) -> str:
        return f"Plan({self.as_dict()})"


class Fault(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int), ("role", ctypes.c_int), ("index", ctypes.c_int),
                ("parity", ctypes.c_int), ("block", ctypes.c_int * 3),
                ("cluster_rank", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_}
        d["block"] = list(self.block)
        return d


_lib = None


def library_path() -> Path:
    return _build.SPLITK_LIB


def load_library():
    """Loads the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not path.exists():
        raise RuntimeError(
            f"{path} is missing: build the sm_103a library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(str(path))
    vp, i, u, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    lib.splitk_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
    lib.splitk_plan.restype = i
    lib.splitk_plan_for.argtypes = [i, i, i, i, i, i, sz, sz, ctypes.POINTER(Plan)]
    lib.splitk_plan_for.restype = i
    lib.splitk_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_bf16.restype = i
    lib.splitk_plan_w4a16_for.argtypes = [i, i, i, i, i, i, sz, sz, ctypes.POINTER(Plan)]
    lib.splitk_plan_w4a16_for.restype = i
    lib.splitk_plan_w4a16.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
    lib.splitk_plan_w4a16.restype = i
    lib.splitk_gemm_w4a16.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_w4a16.restype = i
    lib.splitk_gemm_w4a16_planned.argtypes = [vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(Plan), u, vp]
    lib.splitk_gemm_w4a16_planned.restype = i
    lib.splitk_plan_w8a16_for.argtypes = [i, i, i, i, i, i, sz, sz, ctypes.POINTER(Plan)]
    lib.splitk_plan_w8a16_for.restype = i
    lib.splitk_plan_w8a16.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
    lib.splitk_plan_w8a16.restype = i
    lib.splitk_gemm_w8a16.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_w8a16.restype = i
    lib.splitk_gemm_w8a16_planned.argtypes = [vp, vp, vp, vp, i, i, i, i, ctypes.POINTER(Plan), u, vp]
    lib.splitk_gemm_w8a16_planned.restype = i
    lib.splitk_plan_check_for.argtypes = [ctypes.POINTER(Plan), i, i, i, i, sz, sz]
    lib.splitk_plan_check_for.restype = i
    lib.splitk_plan_candidates_for.argtypes = [i, i, i, i, i, i, sz, sz, ctypes.POINTER(Plan), i]
    lib.splitk_plan_candidates_for.restype = i
    lib.splitk_tune.argtypes = [ctypes.POINTER(vp), i, vp, vp, i, i, i, i, i, i, vp, ctypes.POINTER(Plan),
                                ctypes.POINTER(ctypes.c_float)]
    lib.splitk_tune.restype = i
    lib.splitk_gemm_bf16_bias.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_bf16_bias.restype = i
    lib.splitk_gemm_bf16_planned.argtypes = [vp, vp, vp, i, i, i, i, ctypes.POINTER(Plan), u, vp]
    lib.splitk_gemm_bf16_planned.restype = i
    lib.splitk_gemm_bf16_hostio.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_bf16_hostio.restype = i
    lib.splitk_gemm_bf16_zerocopy.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_bf16_zerocopy.restype = i
    lib.splitk_gemm_bf16_noalloc.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.splitk_gemm_bf16_noalloc.restype = i
    lib.splitk_get_fault.argtypes = [ctypes.POINTER(Fault)]
    lib.splitk_get_fault.restype = i
    lib.splitk_get_status.argtypes = []
    lib.splitk_get_status.restype = i
    lib.splitk_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.splitk_set_wait_limit_ns.restype = i
    lib.splitk_debug_inject.argtypes = [u]
    lib.splitk_debug_inject.restype = i
    lib.splitk_set_trace.argtypes = [vp, sz]
    lib.splitk_set_trace.restype = i
    lib.splitk_release.argtypes = []
    lib.splitk_release.restype = None
    lib.splitk_cache_info.argtypes = [ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(i)]
    lib.splitk_cache_info.restype = i
    lib.splitk_strerror.argtypes = [i]
    lib.splitk_strerror.restype = ctypes.c_char_p
    lib.splitk_version.argtypes = []
    lib.splitk_version.restype = i
    _lib = lib
    return lib


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise SplitKError(rc, where)


# ---------------------------------------------------------------- planning
def splitk_plan(M: int, N: int, K: int, L: int = 1, split_k: int = 0) -> Plan:
    out = Plan()
    _check(load_library().splitk_plan(M, N, K, L, split_k, ctypes.byref(out)), "splitk_plan")
    return out


def splitk_plan_for(M: int, N: int, K: int, L: int, split_k: int, num_sms: int,
                    smem_per_sm: int, smem_per_block_optin: int) -> Plan:
    out = Plan()
    _check(load_library().splitk_plan_for(M, N, K, L, split_k, num_sms, smem_per_sm,
                                          smem_per_block_optin, ctypes.byref(out)),
           "splitk_plan_for")
    return out


# ---------------------------------------------------------------- GEMM
def _dims(a, b):
    import torch
    if a.dim() not in (2, 3) or b.dim() != a.dim():
        raise ValueError("a is [L, N, K] or [N, K]; b is [L, M, K] or [M, K]")
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("a and b must be bfloat16")
    if a.dim() == 2:
        (N, K), (M, Kb), L = a.shape, b.shape, 1
        Lb = 1
    else:
        (L, N, K), (Lb, M, Kb) = a.shape, b.shape
    if K != Kb or L != Lb:
        raise ValueError(f"shape mismatch: a{tuple(a.shape)} b{tuple(b.shape)}")
    return int(M), int(N), int(K), int(L)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream))


def _out(c, a, M, N, L):
    import torch
    shape = (M, N) if a.dim() == 2 else (L, M, N)
    if c is None:
        return torch.empty(shape, dtype=torch.bfloat16, device=a.device)
    if tuple(c.shape) != shape or c.dtype != torch.bfloat16 or not c.is_contiguous():
        raise ValueError(f"c must be a contiguous bfloat16 tensor of shape {shape}")
    if c.device != a.device:
        raise ValueError(f"c must be on {a.device}, the operands' device")
    return c


def _require_cuda(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("operands must be contiguous CUDA tensors")
    if len({str(t.device) for t in ts}) > 1:
        raise ValueError("operands must be on one device")


def splitk_gemm_bf16(a, b, c=None, split_k: int = 0, stream=None):
    """c = b @ a^T (per batch), written once; returns c."""
    import torch
    M, N, K, L = _dims(a, b)
    _require_cuda(a, b)
    c = _out(c, a, M, N, L)
    _require_cuda(c)
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16(
            a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, L, int(split_k),
            _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16")
    return c


WEIGHTS_BF16 = 0
WEIGHTS_E2M1_E8M0 = 1
WEIGHTS_E4M3_E8M0 = 2


def splitk_plan_w4a16_for(M: int, N: int, K: int, L: int, split_k: int, num_sms: int,
                          smem_per_sm: int, smem_per_block_optin: int) -> Plan:
    """The A16W4 plan for a described device (no CUDA)."""
    p = Plan()
    _check(load_library().splitk_plan_w4a16_for(M, N, K, L, split_k, num_sms, smem_per_sm,
                                                smem_per_block_optin, ctypes.byref(p)),
           "splitk_plan_w4a16_for")
    return p


def splitk_plan_w4a16(M: int, N: int, K: int, L: int = 1, split_k: int = 0) -> Plan:
    p = Plan()
    _check(load_library().splitk_plan_w4a16(M, N, K, L, split_k, ctypes.byref(p)), "splitk_plan_w4a16")
    return p


def _w4_dims(a_q, a_s, b):
    import torch
    if a_q.dtype != torch.uint8 or a_s.dtype != torch.uint8:
        raise TypeError("A16W4 codes and scales are uint8 tensors")
    if b.dtype != torch.bfloat16:
        raise TypeError("b must be bfloat16")
    if a_q.dim() not in (2, 3) or a_s.dim() != a_q.dim() or b.dim() != a_q.dim():
        raise ValueError("a_q is [L, N, K/2] or [N, K/2], a_s [L, N, K/32] or [N, K/32], b [L, M, K] or [M, K]")
    if a_q.dim() == 2:
        a_q, a_s = a_q.unsqueeze(0), a_s.unsqueeze(0)
    if b.dim() == 2:
        b = b.unsqueeze(0)
    L, N, K2 = a_q.shape
    K = 2 * K2
    if tuple(a_s.shape) != (L, N, K // 32) or b.shape[0] != L or b.shape[2] != K:
        raise ValueError(f"shape mismatch a_q{tuple(a_q.shape)} a_s{tuple(a_s.shape)} b{tuple(b.shape)}")
    for t in (a_q, a_s, b):
        if not t.is_contiguous():
            raise ValueError("operands must be contiguous")
    return int(b.shape[1]), N, K, L


def splitk_gemm_w4a16(a_q, a_s, b, c=None, split_k: int = 0, stream=None):
    """c = b @ dequant(a_q, a_s)^T (4-bit E2M1 codes, E8M0 scales per 32 k)."""
    import torch
    M, N, K, L = _w4_dims(a_q, a_s, b)
    _require_cuda(a_q, a_s, b)
    c = _out(c, b, M, N, L)
    with torch.cuda.device(b.device):
        rc = load_library().splitk_gemm_w4a16(a_q.data_ptr(), a_s.data_ptr(), b.data_ptr(), c.data_ptr(),
                                              M, N, K, L, int(split_k), _stream_handle(stream, b.device))
    _check(rc, "splitk_gemm_w4a16")
    return c


def splitk_gemm_w4a16_planned(a_q, a_s, b, c, plan: Plan, flags: int = 0, stream=None):
    import torch
    M, N, K, L = _w4_dims(a_q, a_s, b)
    _require_cuda(a_q, a_s, b)
    c = _out(c, b, M, N, L)
    with torch.cuda.device(b.device):
        rc = load_library().splitk_gemm_w4a16_planned(a_q.data_ptr(), a_s.data_ptr(), b.data_ptr(),
                                                      c.data_ptr(), M, N, K, L, ctypes.byref(plan),
                                                      int(flags), _stream_handle(stream, b.device))
    _check(rc, "splitk_gemm_w4a16_planned")
    return c


# ---------------------------------------------------------------- A16W8
def splitk_plan_w8a16_for(M: int, N: int, K: int, L: int, split_k: int, num_sms: int,
                          smem_per_sm: int, smem_per_block_optin: int) -> Plan:
    """The A16W8 plan for a described device (no CUDA)."""
    p = Plan()
    _check(load_library().splitk_plan_w8a16_for(M, N, K, L, split_k, num_sms, smem_per_sm,
                                                smem_per_block_optin, ctypes.byref(p)),
           "splitk_plan_w8a16_for")
    return p


def splitk_plan_w8a16(M: int, N: int, K: int, L: int = 1, split_k: int = 0) -> Plan:
    p = Plan()
    _check(load_library().splitk_plan_w8a16(M, N, K, L, split_k, ctypes.byref(p)), "splitk_plan_w8a16")
    return p


def _w8_dims(a_q, a_s, b):
    import torch
    if a_q.dtype != torch.uint8 or a_s.dtype != torch.uint8:
        raise TypeError("A16W8 codes and scales are uint8 tensors")
    if b.dtype != torch.bfloat16:
        raise TypeError("b must be bfloat16")
    if a_q.dim() not in (2, 3) or a_s.dim() != a_q.dim() or b.dim() != a_q.dim():
        raise ValueError("a_q is [L, N, K] or [N, K], a_s [L, N, K/32] or [N, K/32], b [L, M, K] or [M, K]")
    if a_q.dim() == 2:
        a_q, a_s = a_q.unsqueeze(0), a_s.unsqueeze(0)
    if b.dim() == 2:
        b = b.unsqueeze(0)
    L, N, K = a_q.shape
    if tuple(a_s.shape) != (L, N, K // 32) or b.shape[0] != L or b.shape[2] != K:
        raise ValueError(f"shape mismatch a_q{tuple(a_q.shape)} a_s{tuple(a_s.shape)} b{tuple(b.shape)}")
    for t in (a_q, a_s, b):
        if not t.is_contiguous():
            raise ValueError("operands must be contiguous")
    return int(b.shape[1]), N, K, L


def splitk_gemm_w8a16(a_q, a_s, b, c=None, split_k: int = 0, stream=None):
    """c = b @ dequant(a_q, a_s)^T (8-bit E4M3 codes, E8M0 scales per 32 k)."""
    import torch
    M, N, K, L = _w8_dims(a_q, a_s, b)
    _require_cuda(a_q, a_s, b)
    c = _out(c, b, M, N, L)
    with torch.cuda.device(b.device):
        rc = load_library().splitk_gemm_w8a16(a_q.data_ptr(), a_s.data_ptr(), b.data_ptr(), c.data_ptr(),
                                              M, N, K, L, int(split_k), _stream_handle(stream, b.device))
    _check(rc, "splitk_gemm_w8a16")
    return c


def splitk_gemm_w8a16_planned(a_q, a_s, b, c, plan: Plan, flags: int = 0, stream=None):
    import torch
    M, N, K, L = _w8_dims(a_q, a_s, b)
    _require_cuda(a_q, a_s, b)
    c = _out(c, b, M, N, L)
    with torch.cuda.device(b.device):
        rc = load_library().splitk_gemm_w8a16_planned(a_q.data_ptr(), a_s.data_ptr(), b.data_ptr(),
                                                      c.data_ptr(), M, N, K, L, ctypes.byref(plan),
                                                      int(flags), _stream_handle(stream, b.device))
    _check(rc, "splitk_gemm_w8a16_planned")
    return c


def splitk_plan_check_for(plan: Plan, M: int, N: int, K: int, L: int, smem_per_sm: int,
                          smem_per_block_optin: int) -> int:
    """The launch-time plan check for a described device; returns the status."""
    return load_library().splitk_plan_check_for(ctypes.byref(plan), M, N, K, L, smem_per_sm,
                                                smem_per_block_optin)


def splitk_plan_candidates_for(M: int, N: int, K: int, L: int, split_k: int, num_sms: int,
                               smem_per_sm: int, smem_per_block_optin: int) -> list:
    """Every valid tactic for the shape on a described device (the plan's
    own choice first)."""
    lib = load_library()
    n = lib.splitk_plan_candidates_for(M, N, K, L, split_k, num_sms, smem_per_sm,
                                       smem_per_block_optin, None, 0)
    _check(n if n < 0 else 0, "splitk_plan_candidates_for")
    arr = (Plan * max(n, 1))()
    got = lib.splitk_plan_candidates_for(M, N, K, L, split_k, num_sms, smem_per_sm,
                                         smem_per_block_optin, arr, n)
    _check(got if got < 0 else 0, "splitk_plan_candidates_for")
    return [Plan.from_buffer_copy(arr[k]) for k in range(n)]


def splitk_tune(a_list, b, c=None, split_k: int = 0, reps: int = 64, stream=None):
    """The fastest candidate tactic measured on this device, cycling through
    the same-shape weight tensors `a_list`; returns (plan, us_per_call)."""
    import torch
    M, N, K, L = _dims(a_list[0], b)
    for a in a_list:
        if tuple(a.shape) != tuple(a_list[0].shape) or a.dtype != a_list[0].dtype:
            raise ValueError("the weight tensors must have one shape and dtype")
    _require_cuda(*a_list, b)
    c = _out(c, a_list[0], M, N, L)
    ptrs = (ctypes.c_void_p * len(a_list))(*[a.data_ptr() for a in a_list])
    plan = Plan()
    us = ctypes.c_float(0.0)
    with torch.cuda.device(b.device):
        rc = load_library().splitk_tune(ptrs, len(a_list), b.data_ptr(), c.data_ptr(), M, N, K, L,
                                        int(split_k), int(reps), _stream_handle(stream, b.device),
                                        ctypes.byref(plan), ctypes.byref(us))
    _check(rc, "splitk_tune")
    return plan, float(us.value)


def splitk_gemm_bf16_bias(a, b, bias, c=None, split_k: int = 0, stream=None):
    """c = b @ a^T + bias (bias [L, N] or [N] bfloat16, added in FP32 before
    the one rounding); returns c."""
    import torch
    M, N, K, L = _dims(a, b)
    _require_cuda(a, b, bias)
    if bias.dtype != torch.bfloat16 or bias.numel() != L * N:
        raise ValueError("bias must be a bfloat16 tensor of L*N elements")
    c = _out(c, a, M, N, L)
    _require_cuda(c)
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16_bias(
            a.data_ptr(), b.data_ptr(), bias.data_ptr(), c.data_ptr(), M, N, K, L,
            int(split_k), _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16_bias")
    return c


def splitk_gemm_bf16_noalloc(a, b, c, split_k: int = 0, stream=None):
    """c = b @ a^T through the allocation-free entry point.

    For callers that cannot allocate device memory (see splitk.h): the C
    call allocates nothing, so `c` must be given -- this wrapper does not
    create it either.  Same kernel and results as splitk_gemm_bf16."""
    import torch
    M, N, K, L = _dims(a, b)
    _require_cuda(a, b)
    if c is None:
        raise ValueError("splitk_gemm_bf16_noalloc needs a preallocated output c")
    c = _out(c, a, M, N, L)
    _require_cuda(c)
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16_noalloc(
            a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, L, int(split_k),
            _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16_noalloc")
    return c


def splitk_gemm_bf16_planned(a, b, c, plan: Plan, flags: int = 0, stream=None):
    import torch
    M, N, K, L = _dims(a, b)
    _require_cuda(a, b)
    c = _out(c, a, M, N, L)
    _require_cuda(c)
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16_planned(
            a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, L, ctypes.byref(plan),
            int(flags), _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16_planned")
    return c


def splitk_gemm_bf16_hostio(a, b_host, c_host, b_dev, c_dev, split_k: int = 0, stream=None):
    """Copies b_host -> b_dev, runs the GEMM, copies c_dev -> c_host (all async)."""
    import torch
    M, N, K, L = _dims(a, b_dev)
    _require_cuda(a, b_dev, c_dev)
    if b_host.is_cuda or c_host.is_cuda:
        raise ValueError("b_host and c_host must be host tensors")
    if b_host.numel() != b_dev.numel() or c_host.numel() != c_dev.numel() or \
            c_dev.numel() != L * M * N:
        raise ValueError("host and device buffers must match in size")
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16_hostio(
            a.data_ptr(), b_host.data_ptr(), c_host.data_ptr(), b_dev.data_ptr(),
            c_dev.data_ptr(), M, N, K, L, int(split_k), _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16_hostio")
    return c_host


def splitk_gemm_bf16_zerocopy(a, b_host, c_host, split_k: int = 0, stream=None):
    """c_host = b_host @ a^T with the activations read from, and the output
    written to, pinned host memory by the kernel itself (no copy engines);
    returns c_host.  Synchronize the stream before reading it."""
    import torch
    if b_host.is_cuda or c_host.is_cuda:
        raise ValueError("b_host and c_host must be host tensors")
    _require_cuda(a)
    if a.dtype != torch.bfloat16 or b_host.dtype != torch.bfloat16 or c_host.dtype != torch.bfloat16:
        raise TypeError("a, b_host and c_host must be bfloat16")
    if a.dim() != b_host.dim() or a.dim() not in (2, 3) or not (a.is_contiguous() and b_host.is_contiguous()
                                                                and c_host.is_contiguous()):
        raise ValueError("a and b_host must be contiguous [N, K] and [M, K] (or batched [L, ...])")
    a3 = a if a.dim() == 3 else a.unsqueeze(0)
    b3 = b_host if b_host.dim() == 3 else b_host.unsqueeze(0)
    L, N, K = a3.shape
    if b3.shape[0] != L or b3.shape[2] != K:
        raise ValueError("a and b_host disagree on L or K")
    M = b3.shape[1]
    if c_host.numel() != L * M * N:
        raise ValueError("c_host must hold L * M * N values")
    with torch.cuda.device(a.device):
        rc = load_library().splitk_gemm_bf16_zerocopy(
            a.data_ptr(), b_host.data_ptr(), c_host.data_ptr(), M, N, K, L, int(split_k),
            _stream_handle(stream, a.device))
    _check(rc, "splitk_gemm_bf16_zerocopy")
    return c_host


# ---------------------------------------------------------------- status
def splitk_get_fault() -> dict:
    f = Fault()
    rc = load_library().splitk_get_fault(ctypes.byref(f))
    if rc not in (0, -6):
        raise SplitKError(rc, "splitk_get_fault")
    return f.as_dict()


def splitk_get_status() -> int:
    return int(load_library().splitk_get_status())


def splitk_set_wait_limit_ns(ns: int) -> None:
    _check(load_library().splitk_set_wait_limit_ns(int(ns)), "splitk_set_wait_limit_ns")


def splitk_debug_inject(flags: int) -> None:
    _check(load_library().splitk_debug_inject(int(flags)), "splitk_debug_inject")


def splitk_set_trace(buffer=None) -> None:
    """Trace later launches into `buffer` (a CUDA tensor, 16 uint64 words per
    CTA, see splitk.h); None turns tracing off."""
    if buffer is None:
        _check(load_library().splitk_set_trace(None, 0), "splitk_set_trace")
    else:
        _check(load_library().splitk_set_trace(buffer.data_ptr(),
                                               buffer.numel() * buffer.element_size()),
               "splitk_set_trace")


TRACE_SLOTS = 16
TRACE_FIELDS = ("sm_rank", "start", "synced", "weights_issued", "act_ready", "first_full",
                "last_full", "mma_done", "reduced", "stored", "end", "bar_init", "map_ready",
                "prefetched", "tmem_alloc", "epi_synced")


def splitk_release() -> None:
    load_library().splitk_release()


def splitk_cache_info() -> dict:
    """The memory the library owns on the current CUDA device: device and
    page-locked host bytes of its tensor-map pool, and the maps in it."""
    dev_b, host_b, maps = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    _check(load_library().splitk_cache_info(ctypes.byref(dev_b), ctypes.byref(host_b), ctypes.byref(maps)),
           "splitk_cache_info")
    return {"device_bytes": dev_b.value, "host_bytes": host_b.value, "maps": maps.value}


def splitk_strerror(code: int) -> str:
    return load_library().splitk_strerror(int(code)).decode()


def splitk_version() -> int:
    return int(load_library().splitk_version())
