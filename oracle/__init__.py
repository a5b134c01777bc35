"""ctypes loader for the CPU oracle (``oracle/oracle.cpp``).

Test infrastructure only: the test suite, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg use it. The CUDA library and its Python
binding never import this package.

All wrappers take CPU torch tensors (any strides whose innermost stride is 1)
and work on their bytes, so the oracle sees exactly the bytes the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
_FMT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so with g++ (plain C++17, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off",
               "-shared", "-fPIC", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    """The loaded oracle library.

    ``ORACLE_LIB_OVERRIDE`` (test-only) points at another build of oracle.cpp;
    the mutation tests use it to load copies with planted mistakes.
    """
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIB_OVERRIDE")
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
            L.orc_encode.argtypes = [dbl, i32]
            L.orc_encode.restype = ctypes.c_uint32
            L.orc_decode.argtypes = [ctypes.c_uint32, i32]
            L.orc_decode.restype = dbl
            L.orc_rmsnorm.argtypes = [vp, vp, vp, i64, i64, i64, i64, dbl, i32]
            L.orc_rmsnorm.restype = i32
            L.orc_add_rmsnorm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl, i32]
            L.orc_add_rmsnorm.restype = i32
            L.orc_rope_kv_store.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                            i64, i64, i64, i64, i64, i32, i32]
            L.orc_rope_kv_store.restype = i64
            L.orc_rope_kv_store_style.argtypes = L.orc_rope_kv_store.argtypes + [i32]
            L.orc_rope_kv_store_style.restype = i64
            L.orc_glu.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32]
            L.orc_glu.restype = i32
            L.orc_uclip.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i32, i32, dbl, dbl,
                                    i32]
            L.orc_uclip.restype = i32
            L.orc_paged_decode_attention.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i64, i64, i32,
                                                     i64, dbl, i32]
            L.orc_paged_decode_attention.restype = i64
            L.orc_linear.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32]
            L.orc_linear.restype = i32
            _lib = L
    return _lib


def _cpu(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError(f"oracle: {name} must be a CPU tensor")
    return t


def _row_stride(t: torch.Tensor) -> int:
    if t.dim() == 1:
        return t.shape[0]
    if t.stride(-1) != 1:
        raise ValueError("oracle: innermost stride must be 1")
    return t.stride(-2)


def encode(v: float, fmt: int) -> int:
    return int(lib().orc_encode(float(v), fmt))


def decode(bits: int, fmt: int) -> float:
    return float(lib().orc_decode(int(bits) & 0xFFFFFFFF, fmt))


def rmsnorm(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor, eps: float) -> None:
    """out <- rmsnorm(x) * w, all of one dtype; x and out are [rows, D] views."""
    _cpu(x, "x"), _cpu(w, "w"), _cpu(out, "out")
    rows, D = x.shape
    rc = lib().orc_rmsnorm(x.data_ptr(), w.data_ptr(), out.data_ptr(), rows, D,
                           _row_stride(x), _row_stride(out), float(eps), _FMT[x.dtype])
    if rc != 0:
        raise ValueError("oracle: bad rmsnorm arguments")


def add_rmsnorm(x: torch.Tensor, res: torch.Tensor, w: torch.Tensor, out: torch.Tensor,
                eps: float) -> None:
    """x <- round(x + res) in place; out <- rmsnorm(x) * w."""
    for t, n in ((x, "x"), (res, "res"), (w, "w"), (out, "out")):
        _cpu(t, n)
    rows, D = x.shape
    rc = lib().orc_add_rmsnorm(x.data_ptr(), res.data_ptr(), w.data_ptr(), out.data_ptr(), rows, D,
                               _row_stride(x), _row_stride(res), _row_stride(out), float(eps),
                               _FMT[x.dtype])
    if rc != 0:
        raise ValueError("oracle: bad add_rmsnorm arguments")


def _tok_stride(t: torch.Tensor) -> int:
    # [T, H, D] with the head stride equal to D and unit innermost stride.
    if t.stride(-1) != 1 or t.stride(-2) != t.shape[-1]:
        raise ValueError("oracle: q/k/v must have contiguous heads within a token")
    return t.stride(0)


def rope_kv_store(q, k, v, cos, sin, pos, slot_mapping, kv_cache, max_pos: int | None = None,
                  style: str = "neox") -> int:
    """Rotate q in place, write rotated k and v into kv_cache through slot_mapping.

    style: "neox" pairs (i, i + head_dim/2); "interleaved" (GPT-J) pairs (2i, 2i + 1).
    Returns the error count (bad positions plus out-of-range slots).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (cos, "cos"), (sin, "sin"), (pos, "pos"),
                 (slot_mapping, "slot_mapping"), (kv_cache, "kv_cache")):
        _cpu(t, n)
    assert cos.dtype == torch.float32 and sin.dtype == torch.float32
    assert cos.is_contiguous() and sin.is_contiguous()
    assert pos.dtype == torch.int64 and slot_mapping.dtype == torch.int64
    assert kv_cache.is_contiguous()
    T, n_head, hd = q.shape
    n_kv = k.shape[1]
    _, num_blocks, block_size, _, _ = kv_cache.shape
    if max_pos is None:
        max_pos = cos.shape[0]
    n = lib().orc_rope_kv_store_style(q.data_ptr(), k.data_ptr(), v.data_ptr(), cos.data_ptr(),
                                      sin.data_ptr(), pos.data_ptr(), slot_mapping.data_ptr(),
                                      kv_cache.data_ptr(), T, n_head, n_kv, hd, _tok_stride(q),
                                      _tok_stride(k), _tok_stride(v), int(max_pos), num_blocks,
                                      block_size, _FMT[q.dtype], {"neox": 0, "interleaved": 1}[style])
    if n < 0:
        raise ValueError("oracle: bad rope_kv_store arguments or duplicate slots")
    return int(n)


def glu(gate_up: torch.Tensor, out: torch.Tensor, act: str = "silu") -> None:
    """out[t, j] = act(gate_up[t, j]) * gate_up[t, I + j]; act in {'silu', 'relu'}."""
    _cpu(gate_up, "gate_up"), _cpu(out, "out")
    T, I = out.shape
    rc = lib().orc_glu(gate_up.data_ptr(), out.data_ptr(), T, I, _row_stride(gate_up),
                       _row_stride(out), {"silu": 0, "relu": 1}[act], _FMT[out.dtype])
    if rc != 0:
        raise ValueError("oracle: bad glu arguments")


def swiglu(gate_up, out):
    glu(gate_up, out, "silu")


def reglu(gate_up, out):
    glu(gate_up, out, "relu")


def _nhd(t: torch.Tensor, name: str):
    """(N, H, D, n_stride, h_stride) of a [N, D] or [N, H, D] view with unit innermost stride."""
    if t.stride(-1) != 1 and t.shape[-1] > 1:
        raise ValueError(f"oracle: {name} innermost stride must be 1")
    if t.dim() == 2:
        return t.shape[0], 1, t.shape[1], t.stride(0), t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2], t.stride(0), t.stride(1)
    raise ValueError(f"oracle: {name} must be 2-D or 3-D")


def uclip(x: torch.Tensor, alpha: torch.Tensor, gamma: torch.Tensor, out: torch.Tensor,
          clip_min: float = -1.0, clip_max: float = 1.0) -> None:
    """out <- clamp(alpha * x, clip_min, clip_max) * gamma over the last dimension.

    x and out: [N, D] or [N, H, D] views of one dtype; alpha, gamma: fp32 with 1 (scalar)
    or D (per-channel) entries."""
    for t, n in ((x, "x"), (alpha, "alpha"), (gamma, "gamma"), (out, "out")):
        _cpu(t, n)
    if alpha.dtype != torch.float32 or gamma.dtype != torch.float32:
        raise ValueError("oracle: alpha and gamma are fp32")
    N, H, D, xn, xh = _nhd(x, "x")
    oN, oH, oD, on, oh = _nhd(out, "out")
    if (oN, oH, oD) != (N, H, D) or alpha.numel() not in (1, D) or gamma.numel() not in (1, D):
        raise ValueError("oracle: bad uclip shapes")
    a, g = alpha.contiguous(), gamma.contiguous()
    rc = lib().orc_uclip(x.data_ptr(), a.data_ptr(), g.data_ptr(), out.data_ptr(), N, H, D, xn, xh, on, oh,
                         int(alpha.numel() == D and D > 1), int(gamma.numel() == D and D > 1),
                         float(clip_min), float(clip_max), _FMT[x.dtype])
    if rc != 0:
        raise ValueError("oracle: bad uclip arguments")


def dyht(x, alpha, gamma, out):
    """DyHT: gamma * clamp(alpha * x, -1, 1)."""
    uclip(x, alpha, gamma, out, -1.0, 1.0)


def qk_uclip_rope_kv_store(q, k, v, cos, sin, pos, slot_mapping, kv_cache, q_alpha, q_gamma, k_alpha, k_gamma,
                           clip_min: float = -1.0, clip_max: float = 1.0, max_pos: int | None = None,
                           style: str = "neox") -> int:
    """The Q/K norm followed by RoPE + KV store, as the two oracle operators in sequence.

    Tokens whose position lies in [0, max_pos) get q <- uclip(q) (rounded to the dtype)
    and a normed copy of k; the others are left to rope_kv_store, which leaves their q
    unchanged, caches nothing and counts them. k itself is not modified."""
    if max_pos is None:
        max_pos = cos.shape[0]
    ok = (pos >= 0) & (pos < max_pos)
    kn = k.clone()
    if bool(ok.any()):
        idx = ok.nonzero().flatten()
        qs = q[idx].clone()
        uclip(qs, q_alpha, q_gamma, qs, clip_min, clip_max)
        q[idx] = qs
        ks = kn[idx].clone()
        uclip(ks, k_alpha, k_gamma, ks, clip_min, clip_max)
        kn[idx] = ks
    return rope_kv_store(q, kn, v, cos, sin, pos, slot_mapping, kv_cache, max_pos=max_pos, style=style)


def paged_decode_attention(q, kv_cache, block_table, seq_lens, out, scale: float | None = None) -> int:
    """out[b, h] = softmax(scale * q[b, h] . K) V over request b's cached tokens.

    q, out: [B, n_head, head_dim] (token stride free, heads contiguous); kv_cache:
    contiguous [2, num_blocks, block_size, n_kv_head, head_dim]; block_table: int32
    [B, max_blocks]; seq_lens: int32 [B]. scale defaults to 1 / sqrt(head_dim).
    Returns the count of skipped bad entries."""
    for t, n in ((q, "q"), (kv_cache, "kv_cache"), (block_table, "block_table"), (seq_lens, "seq_lens"),
                 (out, "out")):
        _cpu(t, n)
    assert kv_cache.is_contiguous() and block_table.is_contiguous() and seq_lens.is_contiguous()
    assert block_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    B, n_head, hd = q.shape
    _, num_blocks, block_size, n_kv, _ = kv_cache.shape
    if scale is None:
        scale = 1.0 / float(hd) ** 0.5
    n = lib().orc_paged_decode_attention(q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(),
                                         seq_lens.data_ptr(), out.data_ptr(), B, n_head, n_kv, hd,
                                         _tok_stride(q), _tok_stride(out), num_blocks, block_size,
                                         block_table.shape[1] if block_table.dim() == 2 else 0, float(scale),
                                         _FMT[q.dtype])
    if n < 0:
        raise ValueError("oracle: bad paged_decode_attention arguments")
    return int(n)


def linear(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor) -> None:
    """y[b, n] = sum_k h[b, k] * W[n, k]: h [B, K], W [N, K] contiguous (nn.Linear), y [B, N]."""
    for t, n in ((h, "h"), (W, "W"), (y, "y")):
        _cpu(t, n)
    assert W.is_contiguous()
    B, K = h.shape
    N = W.shape[0]
    rc = lib().orc_linear(h.data_ptr(), W.data_ptr(), y.data_ptr(), B, K, N, _row_stride(h), _row_stride(y),
                          _FMT[h.dtype])
    if rc != 0:
        raise ValueError("oracle: bad linear arguments")


def rmsnorm_linear(x, w_ln, W, y, eps: float) -> None:
    """The norm as the projection's prologue: y = rmsnorm(x) * w_ln @ W^T, with the normed
    rows rounded to the dtype as the separate norm kernel stores them."""
    h = torch.empty(x.shape, dtype=x.dtype)
    rmsnorm(x, w_ln, h, eps)
    linear(h, W, y)


def glu_linear(gate_up, W, y, act: str = "silu") -> None:
    """The GLU as the down projection's prologue: y = (act(gate) * up) @ W^T, the activation
    rounded to the dtype as the separate GLU kernel stores it."""
    B, W2 = gate_up.shape
    h = torch.empty(B, W2 // 2, dtype=gate_up.dtype)
    glu(gate_up, h, act)
    linear(h, W, y)
