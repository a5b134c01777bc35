"""ctypes binding of include/sra.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libsra.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
ACT_CODE = {"silu": 0, "relu": 1}


class SRAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn}: {status_string(status)} (status {status})"
        if status == -8:
            msg += f", cudaError {lib().sra_last_cuda_error()}"
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libsra.so. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` (needs nvcc). There is no fallback implementation.")
            L = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
            L.sra_rmsnorm.argtypes = [vp, vp, vp, i64, i64, i64, i64, f32, i32, vp]
            L.sra_add_rmsnorm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, i32, vp]
            L.sra_rope_kv_store.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i64,
                                            i64, i64, i64, i32, vp, i32, vp]
            L.sra_rope_kv_store_ex.argtypes = L.sra_rope_kv_store.argtypes[:19] + [i32, i32, vp]
            L.sra_rope_kv_store_qk_uclip.argtypes = L.sra_rope_kv_store.argtypes[:19] + [i32, vp, vp, vp, vp, f32,
                                                                                        f32, i32, vp]
            L.sra_paged_decode_attention.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i64, i64, i32,
                                                     i64, f32, vp, i32, vp]
            L.sra_paged_decode_attention_ws.argtypes = L.sra_paged_decode_attention.argtypes[:15] + [vp, i64, vp,
                                                                                                    i32, vp]
            L.sra_paged_decode_attention_noalloc.argtypes = L.sra_paged_decode_attention.argtypes
            L.sra_paged_decode_attention_workspace_size.argtypes = [i64, i32, i32, i32, i64, i32, i32]
            L.sra_paged_decode_attention_workspace_size.restype = i64
            L.sra_linear_workspace_size.argtypes = [i64, i64, i64, i32]
            L.sra_linear_workspace_size.restype = i64
            L.sra_rmsnorm_linear.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, i32, vp]
            L.sra_glu_linear.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, vp]
            L.sra_rmsnorm_linear_ws.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, vp, i64, i32, vp]
            L.sra_glu_linear_ws.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, vp, i64, i32, vp]
            L.sra_glu.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, vp]
            L.sra_swiglu.argtypes = [vp, vp, i64, i64, i64, i64, i32, vp]
            L.sra_uclip.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32, i32, f32, f32, i32,
                                    vp]
            for fn in ("sra_rmsnorm", "sra_add_rmsnorm", "sra_rope_kv_store", "sra_rope_kv_store_ex", "sra_glu",
                       "sra_swiglu", "sra_uclip", "sra_rope_kv_store_qk_uclip", "sra_paged_decode_attention",
                       "sra_rmsnorm_linear", "sra_glu_linear", "sra_paged_decode_attention_ws",
                       "sra_paged_decode_attention_noalloc", "sra_rmsnorm_linear_ws", "sra_glu_linear_ws"):
                getattr(L, fn).restype = i32
            L.sra_status_string.argtypes = [i32]
            L.sra_status_string.restype = ctypes.c_char_p
            L.sra_version.restype = i32
            L.sra_last_cuda_error.restype = i32
            L.sra_wait_timeouts.argtypes = []
            L.sra_wait_timeouts.restype = ctypes.c_uint
            L.sra_wait_selftest.argtypes = [vp, vp]
            L.sra_wait_selftest.restype = i32
            L.sra_set_pdl.argtypes = [i32]
            L.sra_set_pdl.restype = i32
            L.sra_force_variant.argtypes = [ctypes.c_char_p, i32]
            L.sra_force_variant.restype = i32
            L.sra_variant_count.argtypes = [ctypes.c_char_p]
            L.sra_variant_count.restype = i32
            L.sra_variant_name.argtypes = [ctypes.c_char_p, i32]
            L.sra_variant_name.restype = ctypes.c_char_p
            L.sra_pick_variant.argtypes = [ctypes.c_char_p, i64, i64, i64, i64, i32, i32]
            L.sra_pick_variant.restype = i32
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().sra_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise SRAError(fn, status)


def wait_selftest(device="cuda:0") -> int:
    """Run the bounded-wait self-test (about a second) and return what the kernel wrote: 0
    when the wait gave up as it should."""
    r = torch.full((1,), -1, dtype=torch.int32, device=device)
    with torch.cuda.device(r.device):
        _check("sra_wait_selftest", lib().sra_wait_selftest(r.data_ptr(), _stream(r, None)))
    return int(r.item())


def wait_timeouts() -> int:
    """Bounded device waits that ran out on the current device since the library was loaded."""
    return int(lib().sra_wait_timeouts())


def set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch for this thread's later calls; returns the previous setting."""
    return bool(lib().sra_set_pdl(1 if enable else 0))


def force_variant(op: str, variant: int) -> None:
    _check("sra_force_variant", lib().sra_force_variant(op.encode(), int(variant)))


def variant_count(op: str) -> int:
    return int(lib().sra_variant_count(op.encode()))


def variant_name(op: str, variant: int) -> str | None:
    r = lib().sra_variant_name(op.encode(), int(variant))
    return r.decode() if r is not None else None


def pick_variant(op: str, a: int, b: int, c: int = 0, d: int = 0, dtype=torch.bfloat16, num_sms: int = 0) -> int:
    return int(lib().sra_pick_variant(op.encode(), a, b, c, d, DTYPE_CODE[dtype], num_sms))


# --------------------------------------------------------------------- helpers
def _cuda(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in DTYPE_CODE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return DTYPE_CODE[t.dtype]


def _as_rows(t: torch.Tensor, name: str) -> tuple[int, int, int]:
    """(rows, width, row stride) of a [..., width] tensor whose rows share one stride."""
    if t.dim() == 0:
        raise ValueError(f"{name} must have at least one dimension")
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: innermost stride must be 1")
    width = t.shape[-1]
    if t.dim() == 1:
        return 1, width, width
    lead = t.shape[:-1]
    rows = 1
    for s in lead:
        rows *= s
    if rows <= 1:
        return rows, width, max(width, t.stride(-2) if t.dim() >= 2 else width)
    # leading dims must collapse to one uniform row stride
    stride = t.stride(-2)
    expect = stride
    for i in range(t.dim() - 2, -1, -1):
        if t.shape[i] != 1 and t.stride(i) != expect:
            raise ValueError(f"{name}: leading dimensions do not collapse to one row stride")
        expect *= t.shape[i]
    return rows, width, stride


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _same_device(*ts):
    dev = ts[0].device
    for t in ts:
        if t is not None and t.device != dev:
            raise ValueError("all tensors must be on the same CUDA device")


# -------------------------------------------------------------------- operators
def rmsnorm(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None, eps: float = 1e-6,
            stream=None) -> torch.Tensor:
    """out = x * rsqrt(mean(x^2, -1) + eps) * w (fp32 accumulation). out may be x."""
    _cuda(x, "x"), _cuda(w, "w")
    if out is None:
        out = torch.empty_like(x)
    _cuda(out, "out")
    _same_device(x, w, out)
    if w.dtype != x.dtype or out.dtype != x.dtype:
        raise ValueError("x, w and out must share one dtype")
    rows, D, xs = _as_rows(x, "x")
    orows, oD, os_ = _as_rows(out, "out")
    if (orows, oD) != (rows, D) or w.numel() != D or (D > 1 and not w.is_contiguous()):
        raise ValueError("shape mismatch")
    with torch.cuda.device(x.device):
        st = lib().sra_rmsnorm(x.data_ptr(), w.data_ptr(), out.data_ptr(), rows, D, xs, os_, float(eps),
                               _dtype(x), _stream(x, stream))
    _check("sra_rmsnorm", st)
    return out


def add_rmsnorm(x: torch.Tensor, res: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
                eps: float = 1e-6, stream=None) -> torch.Tensor:
    """x <- x + res (in place, rounded to x.dtype); returns out = rmsnorm(x) * w."""
    for t, n in ((x, "x"), (res, "res"), (w, "w")):
        _cuda(t, n)
    if out is None:
        out = torch.empty_like(x)
    _cuda(out, "out")
    _same_device(x, res, w, out)
    if not (res.dtype == w.dtype == out.dtype == x.dtype):
        raise ValueError("x, res, w and out must share one dtype")
    rows, D, xs = _as_rows(x, "x")
    rrows, rD, rs = _as_rows(res, "res")
    orows, oD, os_ = _as_rows(out, "out")
    if (rrows, rD) != (rows, D) or (orows, oD) != (rows, D) or w.numel() != D:
        raise ValueError("shape mismatch")
    with torch.cuda.device(x.device):
        st = lib().sra_add_rmsnorm(x.data_ptr(), res.data_ptr(), w.data_ptr(), out.data_ptr(), rows, D, xs, rs,
                                   os_, float(eps), _dtype(x), _stream(x, stream))
    _check("sra_add_rmsnorm", st)
    return out


def _tok_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 3:
        raise ValueError(f"{name} must be [T, heads, head_dim]")
    if t.numel() == 0:
        return t.shape[1] * t.shape[2]
    if t.stride(-1) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
        raise ValueError(f"{name}: heads must be contiguous within a token")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1] * t.shape[2]


ROPE_STYLE = {"neox": 0, "interleaved": 1}


def rope_kv_store(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cos: torch.Tensor, sin: torch.Tensor,
                  pos: torch.Tensor, slot_mapping: torch.Tensor, kv_cache: torch.Tensor,
                  err_count: torch.Tensor | None = None, max_pos: int | None = None, stream=None,
                  style: str = "neox", qk_uclip=None, clip: tuple[float, float] = (-1.0, 1.0)) -> None:
    """Rotate q in place; write rotated k and v into kv_cache[0/1, slot // bs, slot % bs].

    style: "neox" pairs (i, i + head_dim/2); "interleaved" (GPT-J) pairs (2i, 2i + 1).
    qk_uclip: None, or (q_alpha, q_gamma, k_alpha, k_gamma), fp32 [head_dim] tensors: Q and K
    heads first become clamp(alpha * x, *clip) * gamma (DyHT for the default clip), fused into
    the same kernel."""
    if style not in ROPE_STYLE:
        raise ValueError("style must be 'neox' or 'interleaved'")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cos, "cos"), (sin, "sin"), (pos, "pos"),
                 (slot_mapping, "slot_mapping"), (kv_cache, "kv_cache")):
        _cuda(t, n)
    _same_device(q, k, v, cos, sin, pos, slot_mapping, kv_cache, err_count)
    if not (k.dtype == v.dtype == kv_cache.dtype == q.dtype):
        raise ValueError("q, k, v and kv_cache must share one dtype")
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or not cos.is_contiguous() \
            or not sin.is_contiguous():
        raise ValueError("cos and sin must be contiguous float32 [max_pos, head_dim // 2]")
    if pos.dtype != torch.int64 or slot_mapping.dtype != torch.int64 or not pos.is_contiguous() \
            or not slot_mapping.is_contiguous():
        raise ValueError("pos and slot_mapping must be contiguous int64")
    if kv_cache.dim() != 5 or not kv_cache.is_contiguous() or kv_cache.shape[0] != 2:
        raise ValueError("kv_cache must be contiguous [2, num_blocks, block_size, n_kv_head, head_dim]")
    if err_count is not None:
        _cuda(err_count, "err_count")
        if err_count.dtype != torch.int32:
            raise ValueError("err_count must be int32")
    T, n_head, hd = q.shape
    n_kv = k.shape[1]
    _, nb, bs, cn_kv, chd = kv_cache.shape
    if k.shape != (T, n_kv, hd) or v.shape != (T, n_kv, hd) or (cn_kv, chd) != (n_kv, hd) \
            or pos.numel() != T or slot_mapping.numel() != T:
        raise ValueError("shape mismatch")
    if max_pos is None:
        max_pos = cos.shape[0]
    if cos.shape[-1] != hd // 2 or sin.shape != cos.shape or max_pos > cos.shape[0]:
        raise ValueError("cos / sin tables must be [>= max_pos, head_dim // 2]")
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), cos.data_ptr(), sin.data_ptr(), pos.data_ptr(),
            slot_mapping.data_ptr(), kv_cache.data_ptr(), T, n_head, n_kv, hd, _tok_stride(q, "q"),
            _tok_stride(k, "k"), _tok_stride(v, "v"), int(max_pos), nb, bs,
            err_count.data_ptr() if err_count is not None else None, ROPE_STYLE[style])
    if qk_uclip is None:
        with torch.cuda.device(q.device):
            st = lib().sra_rope_kv_store_ex(*args, _dtype(q), _stream(q, stream))
        _check("sra_rope_kv_store_ex", st)
        return
    params = tuple(qk_uclip)
    if len(params) != 4:
        raise ValueError("qk_uclip is (q_alpha, q_gamma, k_alpha, k_gamma)")
    for t, n in zip(params, ("q_alpha", "q_gamma", "k_alpha", "k_gamma")):
        _cuda(t, n)
        if t.dtype != torch.float32 or t.numel() != hd or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 tensor of head_dim entries")
    _same_device(q, *params)
    with torch.cuda.device(q.device):
        st = lib().sra_rope_kv_store_qk_uclip(*args, *(t.data_ptr() for t in params), float(clip[0]),
                                              float(clip[1]), _dtype(q), _stream(q, stream))
    _check("sra_rope_kv_store_qk_uclip", st)


def glu(gate_up: torch.Tensor, out: torch.Tensor | None = None, act: str = "silu", stream=None) -> torch.Tensor:
    """out[t, j] = act(gate_up[t, j]) * gate_up[t, I + j] for act in {'silu', 'relu'}."""
    _cuda(gate_up, "gate_up")
    rows, W, is_ = _as_rows(gate_up, "gate_up")
    if W % 2:
        raise ValueError("gate_up width must be even (gate | up)")
    I = W // 2
    if out is None:
        out = torch.empty(*gate_up.shape[:-1], I, dtype=gate_up.dtype, device=gate_up.device)
    _cuda(out, "out")
    _same_device(gate_up, out)
    if out.dtype != gate_up.dtype:
        raise ValueError("gate_up and out must share one dtype")
    orows, oI, os_ = _as_rows(out, "out")
    if (orows, oI) != (rows, I):
        raise ValueError("shape mismatch")
    if act not in ACT_CODE:
        raise ValueError("act must be 'silu' or 'relu'")
    with torch.cuda.device(gate_up.device):
        st = lib().sra_glu(gate_up.data_ptr(), out.data_ptr(), rows, I, is_, os_, ACT_CODE[act],
                           _dtype(gate_up), _stream(gate_up, stream))
    _check("sra_glu", st)
    return out


def swiglu(gate_up: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """silu(gate) * up over a fused [.., 2I] gate_up."""
    return glu(gate_up, out, "silu", stream)


def reglu(gate_up: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """relu(gate) * up over a fused [.., 2I] gate_up."""
    return glu(gate_up, out, "relu", stream)


def _nhd(t: torch.Tensor, name: str) -> tuple[int, int, int, int, int]:
    """(N, H, D, n_stride, h_stride) of a [N, D] or [N, H, D] view with unit innermost stride."""
    if t.shape[-1] > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: innermost stride must be 1")
    if t.dim() == 2:
        return t.shape[0], 1, t.shape[1], t.stride(0), t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2], t.stride(0), t.stride(1)
    raise ValueError(f"{name} must be 2-D [N, D] or 3-D [N, H, D]")


def uclip(x: torch.Tensor, alpha: torch.Tensor, gamma: torch.Tensor, out: torch.Tensor | None = None,
          clip_min: float = -1.0, clip_max: float = 1.0, stream=None) -> torch.Tensor:
    """out = clamp(alpha * x, clip_min, clip_max) * gamma over the last dimension.

    x, out: [N, D] or [N, H, D] views (any token and head strides; out may be x for
    in place). alpha, gamma: fp32 with 1 entry (scalar) or D entries (per channel)."""
    _cuda(x, "x")
    _cuda(alpha, "alpha")
    _cuda(gamma, "gamma")
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    _cuda(out, "out")
    _same_device(x, alpha, gamma, out)
    if out.dtype != x.dtype:
        raise ValueError("x and out must share one dtype")
    if alpha.dtype != torch.float32 or gamma.dtype != torch.float32:
        raise ValueError("alpha and gamma must be float32")
    N, H, D, xn, xh = _nhd(x, "x")
    oN, oH, oD, on, oh = _nhd(out, "out")
    if (oN, oH, oD) != (N, H, D):
        raise ValueError("shape mismatch")
    for p, name in ((alpha, "alpha"), (gamma, "gamma")):
        if p.numel() not in (1, D) or (p.numel() > 1 and p.dim() > 0 and p.stride(-1) != 1):
            raise ValueError(f"{name} must hold 1 or D contiguous entries")
    with torch.cuda.device(x.device):
        st = lib().sra_uclip(x.data_ptr(), alpha.data_ptr(), gamma.data_ptr(), out.data_ptr(), N, H, D, xn, xh,
                             on, oh, int(alpha.numel() == D and D > 1), int(gamma.numel() == D and D > 1),
                             float(clip_min), float(clip_max), _dtype(x), _stream(x, stream))
    _check("sra_uclip", st)
    return out


def dyht(x: torch.Tensor, alpha: torch.Tensor, gamma: torch.Tensor, out: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """DyHT: gamma * clamp(alpha * x, -1, 1)."""
    return uclip(x, alpha, gamma, out, -1.0, 1.0, stream)


def decode_attention_workspace(B: int, n_head: int, n_kv_head: int, head_dim: int, max_blocks: int,
                               block_size: int, dtype=torch.bfloat16, device="cuda") -> torch.Tensor | None:
    """A workspace for paged_decode_attention(..., workspace=...), or None when the shape does
    not use one. Reuse it across calls (each call writes what it reads)."""
    n = lib().sra_paged_decode_attention_workspace_size(B, n_head, n_kv_head, head_dim, max_blocks, block_size,
                                                       DTYPE_CODE[dtype])
    if n < 0:
        _check("sra_paged_decode_attention_workspace_size", int(n))
    return torch.zeros(int(n), dtype=torch.uint8, device=device) if n > 0 else None


def _attention_args(q, kv_cache, block_table, seq_lens, out, scale, err_count):
    """Checks and C arguments shared by the decode-attention entry points."""
    for t, n in ((q, "q"), (kv_cache, "kv_cache"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _cuda(t, n)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    _cuda(out, "out")
    _same_device(q, kv_cache, block_table, seq_lens, out, err_count)
    if not (q.dtype == kv_cache.dtype == out.dtype):
        raise ValueError("q, kv_cache and out must share one dtype")
    if kv_cache.dim() != 5 or not kv_cache.is_contiguous() or kv_cache.shape[0] != 2:
        raise ValueError("kv_cache must be contiguous [2, num_blocks, block_size, n_kv_head, head_dim]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [B, max_blocks] tensor")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous int32")
    if err_count is not None:
        _cuda(err_count, "err_count")
        if err_count.dtype != torch.int32:
            raise ValueError("err_count must be int32")
    B, n_head, hd = q.shape
    _, nb, bs, n_kv, chd = kv_cache.shape
    if chd != hd or out.shape != q.shape or block_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / float(hd) ** 0.5
    args = (q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(), B,
            n_head, n_kv, hd, _tok_stride(q, "q"), _tok_stride(out, "out"), nb, bs, block_table.shape[1],
            float(scale))
    err = err_count.data_ptr() if err_count is not None else None
    return out, args, err


def paged_decode_attention(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                           seq_lens: torch.Tensor, out: torch.Tensor | None = None, scale: float | None = None,
                           err_count: torch.Tensor | None = None, stream=None,
                           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """out[b, h] = softmax(scale * q[b, h] . K) V over request b's cached tokens.

    q: [B, n_head, head_dim]; kv_cache: [2, num_blocks, block_size, n_kv_head, head_dim] (the
    layout rope_kv_store writes); block_table: int32 [B, max_blocks]; seq_lens: int32 [B];
    scale defaults to 1 / sqrt(head_dim)."""
    out, args, err = _attention_args(q, kv_cache, block_table, seq_lens, out, scale, err_count)
    with torch.cuda.device(q.device):
        if workspace is None:
            st = lib().sra_paged_decode_attention(*args, err, _dtype(q), _stream(q, stream))
        else:
            _cuda(workspace, "workspace")
            st = lib().sra_paged_decode_attention_ws(*args, workspace.data_ptr(),
                                                     workspace.numel() * workspace.element_size(), err,
                                                     _dtype(q), _stream(q, stream))
    _check("sra_paged_decode_attention" if workspace is None else "sra_paged_decode_attention_ws", st)
    return out


def paged_decode_attention_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                                   seq_lens: torch.Tensor, out: torch.Tensor, scale: float | None = None,
                                   err_count: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_decode_attention for callers that cannot allocate device memory (a serving
    stack whose allocator owns the GPU, a plugin inside another framework): the long-context
    split keeps its partial results in one device array the library holds, so the call
    allocates nothing; `out` is therefore required. Calls on one device share that array:
    order them on one stream. The first call on a device looks up the array's address; make
    it before any stream capture."""
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    out, args, err = _attention_args(q, kv_cache, block_table, seq_lens, out, scale, err_count)
    with torch.cuda.device(q.device):
        st = lib().sra_paged_decode_attention_noalloc(*args, err, _dtype(q), _stream(q, stream))
    _check("sra_paged_decode_attention_noalloc", st)
    return out


def _linear_check(x, W, y, B, K, N):
    _cuda(W, "W")
    if W.dim() != 2 or tuple(W.shape) != (N, K) or not W.is_contiguous():
        raise ValueError("W must be a contiguous [N, K] tensor (nn.Linear's weight)")
    if W.dtype != x.dtype or (y is not None and y.dtype != x.dtype):
        raise ValueError("x, W and y must share one dtype")


def linear_workspace(B: int, K: int, dtype: torch.dtype, device, N: int | None = None) -> torch.Tensor:
    """A workspace for rmsnorm_linear / glu_linear with B rows and K (or I) inputs: B * K elements,
    or, given the output width N, the size the library uses best (room for the tcgen05
    projection's partials where it serves the call)."""
    if N is None:
        return torch.empty(max(1, B * K), dtype=dtype, device=device)
    n = lib().sra_linear_workspace_size(B, K, N, DTYPE_CODE[dtype])
    if n < 0:
        _check("sra_linear_workspace_size", int(n))
    es = torch.empty(0, dtype=dtype).element_size()
    return torch.empty(max(1, -(-int(n) // es)), dtype=dtype, device=device)


def _ws_args(ws, x):
    if ws is None:
        return None, 0
    _cuda(ws, "workspace")
    if ws.dtype != x.dtype:
        raise ValueError("workspace must have x's dtype")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def rmsnorm_linear(x: torch.Tensor, w_ln: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None,
                   eps: float = 1e-6, stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y = rmsnorm(x) * w_ln @ W^T with the norm fused in as the projection's prologue.
    x: [B, K]; w_ln: [K]; W: [N, K] (nn.Linear); y: [B, N]. With a workspace
    (linear_workspace) larger batches run the norm once in its own kernel first
    (sra_rmsnorm_linear_ws)."""
    _cuda(x, "x")
    _cuda(w_ln, "w_ln")
    B, K, xs = _as_rows(x, "x")
    N = W.shape[0]
    _linear_check(x, W, y, B, K, N)
    if w_ln.numel() != K or w_ln.dtype != x.dtype or not w_ln.is_contiguous():
        raise ValueError("w_ln must be a contiguous [K] tensor of x's dtype")
    if y is None:
        y = torch.empty(*x.shape[:-1], N, dtype=x.dtype, device=x.device)
    _cuda(y, "y")
    _same_device(x, w_ln, W, y)
    yr, yn, ys = _as_rows(y, "y")
    if (yr, yn) != (B, N):
        raise ValueError("shape mismatch")
    with torch.cuda.device(x.device):
        if workspace is None:
            st = lib().sra_rmsnorm_linear(x.data_ptr(), w_ln.data_ptr(), W.data_ptr(), y.data_ptr(), B, K, N, xs,
                                          ys, float(eps), _dtype(x), _stream(x, stream))
            _check("sra_rmsnorm_linear", st)
        else:
            _same_device(x, workspace)
            wp, wb = _ws_args(workspace, x)
            st = lib().sra_rmsnorm_linear_ws(x.data_ptr(), w_ln.data_ptr(), W.data_ptr(), y.data_ptr(), B, K, N, xs,
                                             ys, float(eps), wp, wb, _dtype(x), _stream(x, stream))
            _check("sra_rmsnorm_linear_ws", st)
    return y


def glu_linear(gate_up: torch.Tensor, W: torch.Tensor, y: torch.Tensor | None = None, act: str = "silu",
               stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y = (act(gate) * up) @ W^T with the activation fused in as the down projection's prologue.
    gate_up: [B, 2I]; W: [N, I] (nn.Linear); y: [B, N]. With a workspace
    (linear_workspace(B, I, ...)) larger batches run the activation once in its own kernel
    first (sra_glu_linear_ws)."""
    _cuda(gate_up, "gate_up")
    B, W2, xs = _as_rows(gate_up, "gate_up")
    if W2 % 2:
        raise ValueError("gate_up width must be even (gate | up)")
    I = W2 // 2
    N = W.shape[0]
    _linear_check(gate_up, W, y, B, I, N)
    if act not in ACT_CODE:
        raise ValueError("act must be 'silu' or 'relu'")
    if y is None:
        y = torch.empty(*gate_up.shape[:-1], N, dtype=gate_up.dtype, device=gate_up.device)
    _cuda(y, "y")
    _same_device(gate_up, W, y)
    yr, yn, ys = _as_rows(y, "y")
    if (yr, yn) != (B, N):
        raise ValueError("shape mismatch")
    with torch.cuda.device(gate_up.device):
        if workspace is None:
            st = lib().sra_glu_linear(gate_up.data_ptr(), W.data_ptr(), y.data_ptr(), B, I, N, xs, ys, ACT_CODE[act],
                                      _dtype(gate_up), _stream(gate_up, stream))
            _check("sra_glu_linear", st)
        else:
            _same_device(gate_up, workspace)
            wp, wb = _ws_args(workspace, gate_up)
            st = lib().sra_glu_linear_ws(gate_up.data_ptr(), W.data_ptr(), y.data_ptr(), B, I, N, xs, ys,
                                         ACT_CODE[act], wp, wb, _dtype(gate_up), _stream(gate_up, stream))
            _check("sra_glu_linear_ws", st)
    return y
