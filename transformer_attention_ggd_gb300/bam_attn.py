"""Thin ctypes binding of the C ABI in include/bam_attn.h.

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the computation runs in the CUDA kernels
of libbam_attn.so.  There is no fallback: if the library is missing or no
GPU is present, calls raise.

The entry points check every tensor argument (CUDA, current device,
contiguous, the dtype and shape the call implies) before the call and raise
ValueError; ``check=False`` skips that for buffers a caller has already
passed through a checked call (a loop over preallocated tensors).

With BAM_ATTN_DEBUG=1 in the environment the debug build
libbam_attn_debug.so is loaded instead (same ABI; every plain bulk copy and
tiled store is bounds-checked on the device, a failed check is reported by
bam_attn_check_status as BAM_ERR_BOUNDS).

The functions carry the C names (bam_attn_fwd, bam_attn_bwd, ...).  The
helpers at the bottom (``attention_forward`` and friends) allocate outputs
and workspace with torch and then call the same entry points.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
DEBUG = os.environ.get("BAM_ATTN_DEBUG", "0") == "1"
LIB_PATH = os.path.join(PKG, "_build", "libbam_attn_debug.so" if DEBUG else "libbam_attn.so")

BAM_OK = 0
BAM_ERR_INVALID_ARG = 1
BAM_ERR_UNSUPPORTED = 2
BAM_ERR_CUDA = 3
BAM_ERR_TIMEOUT = 4
BAM_ERR_WORKSPACE = 5
BAM_ERR_BOUNDS = 6

BAM_OP_FWD, BAM_OP_BWD, BAM_OP_DECODE = 0, 1, 2
BAM_PRIOR_ALPHA, BAM_PRIOR_THETA = 0, 1

BAM_KERNEL_TABLE = 0
BAM_KERNEL_FWD = 1
BAM_KERNEL_BWD_PREP = 2
BAM_KERNEL_BWD = 3
BAM_KERNEL_BWD_FINAL = 4
BAM_KERNEL_DECODE = 5
BAM_KERNEL_DECODE_COMBINE = 6
BAM_KERNEL_COUNT = 7

# Every symbol that include/bam_attn.h declares.
EXPORTED = (
    "bam_attn_workspace_size",
    "bam_attn_fwd",
    "bam_attn_bwd",
    "bam_attn_decode",
    "bam_attn_decode_varlen",
    "bam_attn_decode_paged",
    "bam_attn_check_status",
    "bam_status_string",
    "bam_attn_profile_events",
    "bam_attn_launch_count",
    "bam_attn_decode_noalloc",
    "bam_attn_decode_noalloc_check_status",
    "bam_attn_selftest_wait",
    "bam_attn_debug_build",
    "bam_attn_debug_arm_giveup",
    "bam_attn_debug_arm_giveup_noalloc",
    "bam_attn_bwd_schedule",
)

# Size of the fixed device scratch of bam_attn_decode_noalloc.
BAM_DECODE_NOALLOC_SCRATCH_BYTES = 4 << 20


class BamError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bam_status_string(status)} (status {status})")


class BamParams(ctypes.Structure):
    _fields_ = [
        ("alpha", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("mu", ctypes.c_void_p),
        ("s", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("causal", ctypes.c_int),
        ("ssmax", ctypes.c_int),
        ("prior", ctypes.c_int),
    ]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libbam_attn.so and declare its signatures (no GPU needed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        pp = ctypes.POINTER(BamParams)
        lib.bam_attn_workspace_size.restype = sz
        lib.bam_attn_workspace_size.argtypes = [i, i, i, i, i]
        lib.bam_attn_fwd.restype = i
        lib.bam_attn_fwd.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, pp, vp, sz, vp]
        lib.bam_attn_bwd.restype = i
        lib.bam_attn_bwd.argtypes = [vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     i, i, i, i, pp, vp, sz, vp]
        lib.bam_attn_decode.restype = i
        lib.bam_attn_decode.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, pp, vp, sz, vp]
        lib.bam_attn_decode_paged.restype = i
        lib.bam_attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, i, i, i, i, i, i, pp,
                                              vp, sz, vp]
        lib.bam_attn_decode_varlen.restype = i
        lib.bam_attn_decode_varlen.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, i, i, pp, vp, sz,
                                               vp]
        lib.bam_attn_check_status.restype = i
        lib.bam_attn_check_status.argtypes = [vp, vp]
        lib.bam_status_string.restype = ctypes.c_char_p
        lib.bam_status_string.argtypes = [i]
        lib.bam_attn_profile_events.restype = i
        lib.bam_attn_profile_events.argtypes = [i, vp, vp]
        lib.bam_attn_launch_count.restype = ctypes.c_uint64
        lib.bam_attn_launch_count.argtypes = []
        lib.bam_attn_decode_noalloc.restype = i
        lib.bam_attn_decode_noalloc.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, pp, vp]
        lib.bam_attn_selftest_wait.restype = i
        lib.bam_attn_selftest_wait.argtypes = [vp, sz, vp]
        lib.bam_attn_debug_build.restype = i
        lib.bam_attn_debug_build.argtypes = []
        lib.bam_attn_decode_noalloc_check_status.restype = i
        lib.bam_attn_decode_noalloc_check_status.argtypes = [vp]
        lib.bam_attn_debug_arm_giveup.restype = i
        lib.bam_attn_debug_arm_giveup.argtypes = [vp, i]
        lib.bam_attn_debug_arm_giveup_noalloc.restype = i
        lib.bam_attn_debug_arm_giveup_noalloc.argtypes = [i]
        ip = ctypes.POINTER(ctypes.c_int)
        lib.bam_attn_bwd_schedule.restype = i
        lib.bam_attn_bwd_schedule.argtypes = [i, i, i, i, i, ip, ip, i]
        _lib = lib
        return lib


# ---------------------------------------------------------------- raw entry points

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_params(alpha, beta, mu, s=None, eps=1e-5, causal=True, ssmax=False,
                prior=BAM_PRIOR_ALPHA) -> BamParams:
    """alpha, beta, mu, s: contiguous float32 CUDA tensors of length H, which
    the returned struct keeps alive.  prior: BAM_PRIOR_ALPHA, or
    BAM_PRIOR_THETA when alpha, beta, mu hold the thetas."""
    import torch
    if not isinstance(alpha, torch.Tensor) or alpha.dim() != 1:
        raise ValueError("alpha must be a 1-D tensor of length H")
    H = alpha.shape[0]
    for name, t in (("alpha", alpha), ("beta", beta), ("mu", mu), ("s", s)):
        _require(t, name, (H,), (torch.float32,), alpha.device, optional=name == "s")
    if ssmax and s is None:
        raise ValueError("ssmax needs the per-head scale s")
    prm = BamParams(alpha.data_ptr(), beta.data_ptr(), mu.data_ptr(),
                    s.data_ptr() if s is not None else None, float(eps), int(bool(causal)),
                    int(bool(ssmax)), int(prior))
    prm.tensors = (alpha, beta, mu, s)
    return prm


# ---------------------------------------------------------------- argument checks
# The C ABI sees raw pointers and sizes only; these checks keep a tensor of
# the wrong shape, dtype, device or layout from reaching the kernels, which
# would read or write outside its storage.

def _require(t, name, shape, dtypes, device, optional=False):
    import torch
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if (t.dtype in dtypes and t.shape == shape and t.is_contiguous()
            and t.device == device):
        return
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _device(q):
    """The CUDA device of q, which must be the current device (the library
    launches there, on that device's stream)."""
    import torch
    if not isinstance(q, torch.Tensor) or not q.is_cuda:
        raise ValueError("q must be a CUDA tensor")
    if q.device.index != torch.cuda.current_device():
        raise ValueError(f"q is on {q.device}, but cuda:{torch.cuda.current_device()} is "
                         "the current device")
    return q.device


_DTYPES = None


def _dt():
    """The dtype tuples the entry points accept: bf16, fp32, an output (fp32
    or bf16) and int32."""
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = ((torch.bfloat16,), (torch.float32,), (torch.float32, torch.bfloat16),
                   (torch.int32,))
    return _DTYPES


def _check_tensors(specs, device):
    """specs: (name, tensor, shape, dtypes, optional) per argument.  One quick
    pass over all of them; only when one fails does the detailed pass run,
    which raises for the first bad argument."""
    for name, t, shape, dtypes, optional in specs:
        if t is None:
            if optional:
                continue
            break
        try:
            if not (t.dtype in dtypes and t.shape == shape and t.is_contiguous()
                    and t.device == device):
                break
        except AttributeError:
            break
    else:
        return
    for name, t, shape, dtypes, optional in specs:
        _require(t, name, shape, dtypes, device, optional)
    raise ValueError("argument check failed")


def _param_specs(params: BamParams, H: int):
    tensors = getattr(params, "tensors", None)
    if tensors is None:
        return ()  # built by hand from raw pointers: the caller vouches for them
    f32 = _dt()[1]
    return tuple((n, t, (H,), f32, n == "s")
                 for n, t in zip(("alpha", "beta", "mu", "s"), tensors))


def _check_ws(ws, device):
    import torch
    if not isinstance(ws, torch.Tensor) or ws.dtype != torch.uint8 or ws.dim() != 1:
        raise ValueError("ws must be a 1-D uint8 tensor (see workspace())")
    if ws.device != device or not ws.is_contiguous():
        raise ValueError(f"ws must be a contiguous tensor on {device}")


def _check(status: int, where: str):
    if status != BAM_OK:
        raise BamError(status, where)


def bam_status_string(status: int) -> str:
    return load_library().bam_status_string(int(status)).decode()


def bam_attn_workspace_size(op: int, B: int, H: int, T: int, D: int = 64) -> int:
    return int(load_library().bam_attn_workspace_size(op, B, H, T, D))


def bam_attn_fwd(q, k, v, o, lse, params: BamParams, ws, stream=None, check=True) -> None:
    import torch
    B, H, T, D = q.shape
    if check:
        dev = _device(q)
        bf, f32, out, _ = _dt()
        x4 = (B, H, T, D)
        _check_tensors((("q", q, x4, bf, False), ("k", k, x4, bf, False), ("v", v, x4, bf, False),
                        ("o", o, x4, out, False), ("lse", lse, (B, H, T), f32, True))
                       + _param_specs(params, H), dev)
        _check_ws(ws, dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), o_fp32, _ptr(lse), B, H,
                                     T, D, ctypes.byref(params), _ptr(ws), ws.numel(),
                                     _stream(stream))
    _check(st, "bam_attn_fwd")


def bam_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, dalpha, dbeta, dmu, ds, params: BamParams,
                 ws, stream=None, check=True) -> None:
    import torch
    B, H, T, D = q.shape
    if check:
        dev = _device(q)
        bf, f32, out, _ = _dt()
        x4 = (B, H, T, D)
        _check_tensors(tuple((n, t, x4, bf, False) for n, t in (
                           ("q", q), ("k", k), ("v", v), ("dO", dO), ("dq", dq), ("dk", dk),
                           ("dv", dv)))
                       + (("o", o, x4, out, False), ("lse", lse, (B, H, T), f32, False))
                       + tuple((n, t, (H,), f32, False) for n, t in (
                           ("dalpha", dalpha), ("dbeta", dbeta), ("dmu", dmu), ("ds", ds)))
                       + _param_specs(params, H), dev)
        _check_ws(ws, dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), o_fp32, _ptr(lse),
                                     _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha),
                                     _ptr(dbeta), _ptr(dmu), _ptr(ds), B, H, T, D,
                                     ctypes.byref(params), _ptr(ws), ws.numel(),
                                     _stream(stream))
    _check(st, "bam_attn_bwd")


def _decode_specs(q, o, lse, B, H, D):
    bf, f32, out, _ = _dt()
    return (("q", q, (B, H, D), bf, False), ("o", o, (B, H, D), out, False),
            ("lse", lse, (B, H), f32, True))


def bam_attn_decode(q, kc, vc, o, lse, params: BamParams, ws, stream=None, check=True) -> None:
    import torch
    B, H, Tkv, D = kc.shape
    if check:
        dev = _device(q)
        bf = _dt()[0]
        kv = (B, H, Tkv, D)
        _check_tensors((("kc", kc, kv, bf, False), ("vc", vc, kv, bf, False))
                       + _decode_specs(q, o, lse, B, H, D) + _param_specs(params, H), dev)
        _check_ws(ws, dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(o), o_fp32, _ptr(lse),
                                        B, H, Tkv, D, ctypes.byref(params), _ptr(ws), ws.numel(),
                                        _stream(stream))
    _check(st, "bam_attn_decode")


def bam_attn_decode_varlen(q, kc, vc, cache_lens, o, lse, params: BamParams, ws,
                           stream=None, check=True) -> None:
    """cache_lens: int32 CUDA tensor [B] (each in [1, Tmax]); kc, vc: [B,H,Tmax,64]."""
    import torch
    B, H, Tmax, D = kc.shape
    if check:
        dev = _device(q)
        bf, _, _, i32 = _dt()
        _check_tensors((("kc", kc, (B, H, Tmax, D), bf, False),
                        ("vc", vc, (B, H, Tmax, D), bf, False),
                        ("cache_lens", cache_lens, (B,), i32, False))
                       + _decode_specs(q, o, lse, B, H, D) + _param_specs(params, H), dev)
        _check_ws(ws, dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_decode_varlen(_ptr(q), _ptr(kc), _ptr(vc), _ptr(cache_lens),
                                               _ptr(o), o_fp32, _ptr(lse), B, H, Tmax, D,
                                               ctypes.byref(params), _ptr(ws), ws.numel(),
                                               _stream(stream))
    _check(st, "bam_attn_decode_varlen")


def bam_attn_decode_paged(q, k_pages, v_pages, block_table, cache_lens, o, lse,
                          params: BamParams, ws, stream=None, check=True) -> None:
    """k_pages, v_pages: [num_pages, H, page, 64]; block_table int32 [B, max_blocks];
    cache_lens int32 [B]."""
    import torch
    num_pages, H, page, D = k_pages.shape
    B, max_blocks = block_table.shape
    if check:
        dev = _device(q)
        bf, _, _, i32 = _dt()
        pages = (num_pages, H, page, D)
        _check_tensors((("k_pages", k_pages, pages, bf, False),
                        ("v_pages", v_pages, pages, bf, False),
                        ("block_table", block_table, (B, max_blocks), i32, False),
                        ("cache_lens", cache_lens, (B,), i32, False))
                       + _decode_specs(q, o, lse, B, H, D) + _param_specs(params, H), dev)
        _check_ws(ws, dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages),
                                              _ptr(block_table), _ptr(cache_lens), _ptr(o),
                                              o_fp32, _ptr(lse), B, H, page, max_blocks,
                                              num_pages, D, ctypes.byref(params), _ptr(ws),
                                              ws.numel(), _stream(stream))
    _check(st, "bam_attn_decode_paged")


def bam_attn_decode_noalloc(q, kc, vc, o, lse, params: BamParams, stream=None,
                            check=True) -> None:
    """Decode for callers that cannot allocate device memory (plugin-style
    hosts that only pass input/output pointers; loops that cannot afford
    cudaMalloc's possible synchronisation): no workspace argument, scratch
    from the library's fixed device array.  Overlapping calls race."""
    import torch
    B, H, Tkv, D = kc.shape
    if check:
        dev = _device(q)
        bf = _dt()[0]
        kv = (B, H, Tkv, D)
        _check_tensors((("kc", kc, kv, bf, False), ("vc", vc, kv, bf, False))
                       + _decode_specs(q, o, lse, B, H, D) + _param_specs(params, H), dev)
    o_fp32 = 1 if o.dtype == torch.float32 else 0
    st = load_library().bam_attn_decode_noalloc(_ptr(q), _ptr(kc), _ptr(vc), _ptr(o), o_fp32,
                                                _ptr(lse), B, H, Tkv, D, ctypes.byref(params),
                                                _stream(stream))
    _check(st, "bam_attn_decode_noalloc")


def bam_attn_selftest_wait(ws, stream=None) -> None:
    """Launch the failure-detection self-test: a bounded wait that runs out
    and records BAM_ERR_TIMEOUT in the status word of `ws` (about 2 s)."""
    _check(load_library().bam_attn_selftest_wait(_ptr(ws), ws.numel(), _stream(stream)),
           "bam_attn_selftest_wait")


def bam_attn_check_status(ws, stream=None) -> int:
    return int(load_library().bam_attn_check_status(_ptr(ws), _stream(stream)))


def bam_attn_decode_noalloc_check_status(stream=None) -> int:
    """Status of the no-alloc decode calls on the current device since the
    previous check (synchronises the stream; reads and clears)."""
    return int(load_library().bam_attn_decode_noalloc_check_status(_stream(stream)))


def bam_attn_debug_build() -> bool:
    """True when the loaded library is the bounds-checking debug build."""
    return bool(load_library().bam_attn_debug_build())


def bam_attn_debug_arm_giveup(ws, n: int) -> int:
    """Debug build: the n-th bounded device wait of the next calls on `ws`
    gives up (0 disarms).  Returns the status (BAM_ERR_UNSUPPORTED in the
    release build)."""
    return int(load_library().bam_attn_debug_arm_giveup(_ptr(ws), int(n)))


def bam_attn_debug_arm_giveup_noalloc(n: int) -> int:
    """As bam_attn_debug_arm_giveup, for the no-alloc decode's scratch."""
    return int(load_library().bam_attn_debug_arm_giveup_noalloc(int(n)))


def bam_attn_profile_events(which: int, before=None, after=None) -> None:
    b = ctypes.c_void_p(before.cuda_event) if before is not None else None
    a = ctypes.c_void_p(after.cuda_event) if after is not None else None
    _check(load_library().bam_attn_profile_events(which, b, a), "bam_attn_profile_events")


def bam_attn_launch_count() -> int:
    return int(load_library().bam_attn_launch_count())


def bam_attn_bwd_schedule(B: int, H: int, T: int, causal: bool, grid: int):
    """The causal backward's per-CTA item lists for `grid` CTAs (host only):
    a list of item-index lists, CTA by CTA, or None when the kernel deals
    items out round-robin itself.  Item w is key tile w // (B*H) of
    (b, h) = w % (B*H)."""
    nkb = (T + 127) // 128
    total = nkb * B * H
    g = min(grid, total)
    start = (ctypes.c_int * (g + 1))()
    item = (ctypes.c_int * max(total, 1))()
    n = int(load_library().bam_attn_bwd_schedule(int(B), int(H), int(T), int(bool(causal)),
                                                 int(grid), start, item, total))
    if n < 0:
        raise BamError(BAM_ERR_INVALID_ARG, "bam_attn_bwd_schedule")
    if n == 0:
        return None
    return [list(item[start[c]:start[c + 1]]) for c in range(g)]


# ---------------------------------------------------------------- allocating helpers

def workspace(op: int, B: int, H: int, T: int, device="cuda"):
    import torch
    n = bam_attn_workspace_size(op, B, H, T, 64)
    if n == 0:
        raise BamError(BAM_ERR_INVALID_ARG, "bam_attn_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def attention_forward(q, k, v, alpha, beta, mu, s=None, eps=1e-5, causal=True, ssmax=False,
                      o_dtype=None, ws=None, stream=None, prior=BAM_PRIOR_ALPHA):
    """q, k, v: bf16 [B,H,T,64] CUDA tensors -> (o, lse).  With
    prior=BAM_PRIOR_THETA, alpha, beta, mu are theta_alpha, theta_beta, theta_mu."""
    import torch
    B, H, T, D = q.shape
    o = torch.empty((B, H, T, D), dtype=o_dtype or torch.float32, device=q.device)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(BAM_OP_FWD, B, H, T, q.device)
    prm = make_params(alpha, beta, mu, s, eps, causal, ssmax, prior)
    bam_attn_fwd(q, k, v, o, lse, prm, ws, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dO, alpha, beta, mu, s=None, eps=1e-5, causal=True,
                       ssmax=False, ws=None, stream=None, prior=BAM_PRIOR_ALPHA):
    """Returns dq, dk, dv (bf16) and dalpha, dbeta, dmu, ds (fp32 [H]); with
    prior=BAM_PRIOR_THETA the three prior gradients are the thetas'."""
    import torch
    B, H, T, D = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    g = [torch.empty(H, dtype=torch.float32, device=q.device) for _ in range(4)]
    if ws is None:
        ws = workspace(BAM_OP_BWD, B, H, T, q.device)
    prm = make_params(alpha, beta, mu, s, eps, causal, ssmax, prior)
    bam_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, g[0], g[1], g[2], g[3], prm, ws, stream)
    return dq, dk, dv, g[0], g[1], g[2], g[3]


def attention_decode(q, kc, vc, alpha, beta, mu, s=None, eps=1e-5, ssmax=False, o_dtype=None,
                     ws=None, stream=None, prior=BAM_PRIOR_ALPHA):
    """q: bf16 [B,H,64]; kc, vc: bf16 [B,H,Tkv,64] -> (o [B,H,64], lse [B,H])."""
    import torch
    B, H, Tkv, D = kc.shape
    o = torch.empty((B, H, D), dtype=o_dtype or torch.float32, device=q.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(BAM_OP_DECODE, B, H, Tkv, q.device)
    prm = make_params(alpha, beta, mu, s, eps, True, ssmax, prior)
    bam_attn_decode(q, kc, vc, o, lse, prm, ws, stream)
    return o, lse


def attention_decode_varlen(q, kc, vc, cache_lens, alpha, beta, mu, s=None, eps=1e-5,
                            ssmax=False, o_dtype=None, ws=None, stream=None,
                            prior=BAM_PRIOR_ALPHA):
    """Ragged decode: q bf16 [B,H,64]; kc, vc bf16 [B,H,Tmax,64]; cache_lens
    int32 [B] -> (o [B,H,64], lse [B,H])."""
    import torch
    B, H, Tmax, D = kc.shape
    o = torch.empty((B, H, D), dtype=o_dtype or torch.float32, device=q.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(BAM_OP_DECODE, B, H, Tmax, q.device)
    prm = make_params(alpha, beta, mu, s, eps, True, ssmax, prior)
    bam_attn_decode_varlen(q, kc, vc, cache_lens, o, lse, prm, ws, stream)
    return o, lse


def attention_decode_paged(q, k_pages, v_pages, block_table, cache_lens, alpha, beta, mu,
                           s=None, eps=1e-5, ssmax=False, o_dtype=None, ws=None, stream=None,
                           prior=BAM_PRIOR_ALPHA):
    """Paged decode: q bf16 [B,H,64]; k_pages, v_pages bf16 [num_pages,H,page,64];
    block_table int32 [B, max_blocks]; cache_lens int32 [B] -> (o, lse)."""
    import torch
    B, H, D = q.shape
    page, max_blocks = k_pages.shape[2], block_table.shape[1]
    o = torch.empty((B, H, D), dtype=o_dtype or torch.float32, device=q.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(BAM_OP_DECODE, B, H, page * max_blocks, q.device)
    prm = make_params(alpha, beta, mu, s, eps, True, ssmax, prior)
    bam_attn_decode_paged(q, k_pages, v_pages, block_table, cache_lens, o, lse, prm, ws, stream)
    return o, lse
