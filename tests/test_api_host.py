"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function include/sra.h declares, and
reject every invalid argument with its status code before making any CUDA
call. Fake addresses are only ever passed together with an argument that is
invalid, so no call here can reach a kernel launch even on a GPU machine.
"""
import ctypes
import os
import re

import pytest

import swiglu_rmsnorm_add_gb300 as sra
from swiglu_rmsnorm_add_gb300 import build as sra_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sra.h")

OK, NULL, SHAPE, STRIDE, DTYPE, ALIAS, ARG, VARIANT = 0, -1, -2, -3, -4, -5, -6, -7
BF16, F16, F32 = 2, 1, 0
P = 0x10000  # a fake, never dereferenced device address


@pytest.fixture(scope="module")
def L():
    sra_build.build()
    return sra.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SRA_API\s+[\w\s\*]*?\b(sra_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("sra_rmsnorm", "sra_add_rmsnorm", "sra_rope_kv_store", "sra_rope_kv_store_ex", "sra_glu",
              "sra_swiglu", "sra_uclip", "sra_paged_decode_attention", "sra_rope_kv_store_qk_uclip",
              "sra_rmsnorm_linear", "sra_glu_linear", "sra_paged_decode_attention_ws",
              "sra_paged_decode_attention_workspace_size", "sra_paged_decode_attention_noalloc",
              "sra_linear_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    # and nothing else (the static CUDA runtime stays hidden)
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", sra_build.LIB], capture_output=True, text=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert exported == declared_functions()


def test_version_and_strings(L):
    assert L.sra_version() == 1
    for code in range(-9, 1):
        assert sra.status_string(code)
    assert sra.status_string(-1234) == "unknown status"


def test_rmsnorm_validation(L):
    f = L.sra_rmsnorm
    assert f(P, P, P + 4096, 4, 16, 16, 16, 1e-6, 7, None) == DTYPE
    assert f(P, P, P + 4096, -1, 16, 16, 16, 1e-6, BF16, None) == SHAPE
    assert f(P, P, P + 4096, 4, 0, 16, 16, 1e-6, BF16, None) == SHAPE
    assert f(P, P, P + 4096, 4, 16, 15, 16, 1e-6, BF16, None) == STRIDE
    assert f(P, P, P + 4096, 4, 16, 16, 8, 1e-6, BF16, None) == STRIDE
    assert f(P, P, P + 4096, 4, 16, 16, 16, -1.0, BF16, None) == ARG
    assert f(P, P, P + 4096, 4, 16, 16, 16, float("nan"), BF16, None) == ARG
    assert f(None, P, P + 4096, 4, 16, 16, 16, 1e-6, BF16, None) == NULL
    assert f(P, None, P + 4096, 4, 16, 16, 16, 1e-6, BF16, None) == NULL
    assert f(P, P + 8192, None, 4, 16, 16, 16, 1e-6, BF16, None) == NULL
    # zero rows: a valid no-op, even with NULL pointers
    assert f(None, None, None, 0, 16, 16, 16, 1e-6, BF16, None) == OK
    # out overlapping x without being x, and out overlapping w
    assert f(P, P + 8192, P + 2, 4, 16, 16, 16, 1e-6, BF16, None) == ALIAS
    assert f(P, P + 4096, P + 4096 + 16, 4, 16, 16, 16, 1e-6, BF16, None) == ALIAS
    # in place with a different stride is not the same view
    assert f(P, P + 8192, P, 4, 16, 16, 32, 1e-6, BF16, None) == ALIAS


def test_add_rmsnorm_validation(L):
    f = L.sra_add_rmsnorm
    X, R, W, O = P, P + 4096, P + 8192, P + 12288
    assert f(X, None, W, O, 4, 16, 16, 16, 16, 1e-6, BF16, None) == NULL
    assert f(X, R, W, O, 4, 16, 16, 8, 16, 1e-6, BF16, None) == STRIDE
    assert f(X, R, W, X, 4, 16, 16, 16, 16, 1e-6, BF16, None) == ALIAS       # out == x forbidden
    assert f(X, R, W, R, 4, 16, 16, 16, 16, 1e-6, BF16, None) == ALIAS       # out == res
    assert f(X, R, W, W, 4, 16, 16, 16, 16, 1e-6, BF16, None) == ALIAS       # out == w
    assert f(X, X + 2, W, O, 4, 16, 16, 16, 16, 1e-6, BF16, None) == ALIAS   # res overlaps x
    assert f(X, R, W, O, 0, 16, 16, 16, 16, 1e-6, BF16, None) == OK


def test_rope_validation(L):
    f = L.sra_rope_kv_store
    Q, K, V, C, S, PO, SL, KV = (P + i * 0x100000 for i in range(8))

    def call(**kw):
        a = dict(q=Q, k=K, v=V, cos=C, sin=S, pos=PO, slot=SL, cache=KV, T=4, nh=12, nkv=2, hd=128,
                 qs=1536, ks=256, vs=256, max_pos=32768, nb=16, bs=16, err=None, dt=BF16)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["cos"], a["sin"], a["pos"], a["slot"], a["cache"], a["T"], a["nh"],
                 a["nkv"], a["hd"], a["qs"], a["ks"], a["vs"], a["max_pos"], a["nb"], a["bs"], a["err"],
                 a["dt"], None)

    assert call(dt=3) == DTYPE
    assert call(T=-1) == SHAPE
    assert call(nh=12, nkv=5) == SHAPE
    assert call(hd=127, qs=12 * 127, ks=2 * 127, vs=2 * 127) == SHAPE
    assert call(bs=0) == SHAPE
    assert call(nb=-1) == SHAPE
    assert call(max_pos=-5) == SHAPE
    assert call(qs=1535) == STRIDE
    assert call(ks=255) == STRIDE
    assert call(vs=100) == STRIDE
    for name in ("q", "k", "v", "cos", "sin", "pos", "slot", "cache"):
        assert call(**{name: None}) == NULL, name
    assert call(T=0) == OK
    assert call(k=Q + 64) == ALIAS                 # q overlaps k
    assert call(cache=V + 2) == ALIAS              # cache overlaps v


def test_rope_style_validation(L):
    """sra_rope_kv_store_ex: the style is checked with the other arguments; the
    neox entry point is the same call with style 0."""
    f = L.sra_rope_kv_store_ex
    Q, K, V, C, S, PO, SL, KV = (P + i * 0x100000 for i in range(8))

    def call(style, T=4, dt=BF16, q=Q):
        return f(q, K, V, C, S, PO, SL, KV, T, 12, 2, 128, 1536, 256, 256, 32768, 16, 16, None, style, dt, None)

    for style in (-1, 2, 7):
        assert call(style) == ARG, style
    assert call(1, dt=3) == DTYPE
    assert call(1, T=-1) == SHAPE
    assert call(1, q=None) == NULL
    assert call(1, T=0) == OK
    assert call(0, T=0) == OK
    with pytest.raises(ValueError):
        sra.rope_kv_store(*([None] * 8), style="gptj")


def test_rope_qk_uclip_validation(L):
    f = L.sra_rope_kv_store_qk_uclip
    Q, K, V, C, S, PO, SL, KV, QA, QG, KA, KG = (P + i * 0x100000 for i in range(12))

    def call(**kw):
        a = dict(q=Q, cache=KV, T=4, style=0, qa=QA, qg=QG, ka=KA, kg=KG, lo=-1.0, hi=1.0, dt=BF16)
        a.update(kw)
        return f(a["q"], K, V, C, S, PO, SL, a["cache"], a["T"], 12, 2, 128, 1536, 256, 256, 32768, 16, 16, None,
                 a["style"], a["qa"], a["qg"], a["ka"], a["kg"], a["lo"], a["hi"], a["dt"], None)

    assert call(lo=1.0, hi=0.0) == ARG
    assert call(hi=float("nan")) == ARG
    assert call(style=3) == ARG
    assert call(dt=9) == DTYPE
    for name in ("qa", "qg", "ka", "kg"):
        assert call(**{name: None}) == NULL, name
    assert call(qa=Q + 64) == ALIAS              # a parameter array inside q
    assert call(kg=KV + 64) == ALIAS             # ... or inside the cache
    assert call(T=0) == OK


def test_paged_decode_attention_validation(L):
    f = L.sra_paged_decode_attention
    Q, C, TB, SL, O, E = (P + i * 0x1000000 for i in range(6))

    def call(**kw):
        a = dict(q=Q, c=C, tb=TB, sl=SL, o=O, B=4, nh=12, nkv=2, hd=128, qs=1536, os=1536, nb=64, bs=16, mb=8,
                 scale=0.088, dt=BF16)
        a.update(kw)
        return f(a["q"], a["c"], a["tb"], a["sl"], a["o"], a["B"], a["nh"], a["nkv"], a["hd"], a["qs"], a["os"],
                 a["nb"], a["bs"], a["mb"], a["scale"], None, a["dt"], None)

    assert call(dt=4) == DTYPE
    assert call(B=-1) == SHAPE
    assert call(nh=12, nkv=5) == SHAPE
    assert call(nh=18, nkv=2) == SHAPE            # 9 query heads per kv head
    assert call(hd=96, qs=12 * 96, os=12 * 96) == SHAPE
    assert call(bs=12) == SHAPE
    assert call(nb=-1) == SHAPE
    assert call(mb=-1) == SHAPE
    assert call(qs=1535) == STRIDE
    assert call(os=100) == STRIDE
    assert call(scale=float("inf")) == ARG
    assert call(scale=float("nan")) == ARG
    for name in ("q", "c", "tb", "sl", "o"):
        assert call(**{name: None}) == NULL, name
    assert call(c=C + 8) == ARG                   # cache not 16-byte aligned
    assert call(o=Q + 64) == ALIAS               # out overlapping q
    assert call(o=C + 1024) == ALIAS             # out inside the cache
    assert call(o=TB) == ALIAS
    assert call(B=0) == OK


def test_linear_validation(L):
    X, WL, W, Y = (P + i * 0x1000000 for i in range(4))
    f = L.sra_rmsnorm_linear
    assert f(X, WL, W, Y, 4, 64, 64, 64, 64, 1e-6, 7, None) == DTYPE
    assert f(X, WL, W, Y, -1, 64, 64, 64, 64, 1e-6, BF16, None) == SHAPE
    assert f(X, WL, W, Y, 4, 0, 64, 64, 64, 1e-6, BF16, None) == SHAPE
    assert f(X, WL, W, Y, 4, 64, 0, 64, 64, 1e-6, BF16, None) == SHAPE
    assert f(X, WL, W, Y, 4, 64, 64, 63, 64, 1e-6, BF16, None) == STRIDE
    assert f(X, WL, W, Y, 4, 64, 64, 64, 63, 1e-6, BF16, None) == STRIDE
    assert f(X, WL, W, Y, 4, 64, 64, 64, 64, -1.0, BF16, None) == ARG
    assert f(X, None, W, Y, 4, 64, 64, 64, 64, 1e-6, BF16, None) == NULL
    assert f(X, WL, None, Y, 4, 64, 64, 64, 64, 1e-6, BF16, None) == NULL
    assert f(X, WL, W, X + 64, 4, 64, 64, 64, 64, 1e-6, BF16, None) == ALIAS
    assert f(X, WL, W, W + 64, 4, 64, 64, 64, 64, 1e-6, BF16, None) == ALIAS
    assert f(X, WL, W, Y, 0, 64, 64, 64, 64, 1e-6, BF16, None) == OK
    g = L.sra_glu_linear
    assert g(X, W, Y, 4, 64, 64, 128, 64, 2, BF16, None) == ARG
    assert g(X, W, Y, 4, 64, 64, 127, 64, 0, BF16, None) == STRIDE
    assert g(X, W, X + 200, 4, 64, 64, 128, 64, 0, BF16, None) == ALIAS
    assert g(None, W, Y, 4, 64, 64, 128, 64, 0, BF16, None) == NULL
    assert g(X, W, Y, 0, 64, 64, 128, 64, 1, BF16, None) == OK


def test_linear_workspace_validation(L):
    X, WL, W, Y, WS = (P + i * 0x1000000 for i in range(5))
    f = L.sra_rmsnorm_linear_ws
    # the fused call's checks come first, nothing runs on error
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, WS, 1 << 20, 7, None) == DTYPE
    assert f(X, WL, W, Y, 64, 64, 64, 63, 64, 1e-6, WS, 1 << 20, BF16, None) == STRIDE
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, WS, -1, BF16, None) == ARG
    assert f(X, None, W, Y, 64, 64, 64, 64, 64, 1e-6, WS, 1 << 20, BF16, None) == NULL
    # from 32 rows the workspace must hold B * K elements and overlap nothing
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, WS, 64 * 64 * 2 - 2, BF16, None) == ARG
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, X + 64, 1 << 20, BF16, None) == ALIAS
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, W, 1 << 20, BF16, None) == ALIAS
    assert f(X, WL, W, Y, 64, 64, 64, 64, 64, 1e-6, Y, 1 << 20, BF16, None) == ALIAS
    assert f(X, WL, W, X + 64, 64, 64, 64, 64, 64, 1e-6, WS, 1 << 20, BF16, None) == ALIAS
    assert f(X, WL, W, Y, 0, 64, 64, 64, 64, 1e-6, WS, 0, BF16, None) == OK
    g = L.sra_glu_linear_ws
    assert g(X, W, Y, 64, 64, 64, 128, 64, 2, WS, 1 << 20, BF16, None) == ARG
    assert g(X, W, Y, 64, 64, 64, 128, 64, 0, WS, 64 * 64 * 2 - 2, BF16, None) == ARG
    assert g(X, W, Y, 64, 64, 64, 128, 64, 0, X + 128, 1 << 20, BF16, None) == ALIAS
    assert g(X, W, Y, 0, 64, 64, 128, 64, 1, WS, 0, BF16, None) == OK


def test_linear_workspace_size(L):
    f = L.sra_linear_workspace_size
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
    f.restype = ctypes.c_int64
    h = (64 * 8960 * 2 + 255) // 256 * 256
    # up to 64 rows and N a multiple of 128 (the tcgen05 projection): h, then [N / 128][16][64][128] fp32
    assert f(64, 8960, 1536, BF16) == h + 1536 // 128 * 16 * 64 * 128 * 4
    assert f(65, 8960, 1536, BF16) == (65 * 8960 * 2 + 255) // 256 * 256
    assert f(64, 8960, 1600, BF16) == h
    assert f(64, 8960, 1536, 0) == (64 * 8960 * 4 + 255) // 256 * 256   # fp32 takes no tensor cores
    assert f(0, 8960, 1536, BF16) == 1536 // 128 * 16 * 64 * 128 * 4
    assert f(64, 8960, 1536, 9) == DTYPE
    assert f(-1, 8960, 1536, BF16) == SHAPE


def test_attention_workspace_validation(L):
    f = L.sra_paged_decode_attention_workspace_size
    assert f(1, 12, 2, 128, 2048, 16, 9) == DTYPE
    assert f(-1, 12, 2, 128, 2048, 16, BF16) == SHAPE
    assert f(1, 18, 2, 128, 2048, 16, BF16) == SHAPE
    assert f(1, 12, 2, 96, 2048, 16, BF16) == SHAPE
    assert f(1, 12, 2, 128, 2048, 16, F32) == 0          # the fp32 kernel takes no workspace
    assert f(1, 12, 2, 256, 2048, 16, BF16) == 0         # nor head_dim 256
    assert f(0, 12, 2, 128, 2048, 16, BF16) == 0
    g = L.sra_paged_decode_attention_ws
    Q, C, TB, SL, O = (P + i * 0x1000000 for i in range(5))
    assert g(Q, C, TB, SL, O, 4, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, -1, None, BF16, None) == ARG
    assert g(Q, C, TB, SL, O, 4, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, 0, None, 7, None) == DTYPE
    assert g(Q, C, TB, SL, O, 0, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, 0, None, BF16, None) == OK


def test_attention_noalloc_validation(L):
    # the library-held scratch variant rejects what the other entry points reject, before
    # touching a device
    h = L.sra_paged_decode_attention_noalloc
    Q, C, TB, SL, O = (P + i * 0x1000000 for i in range(5))
    assert h(Q, C, TB, SL, O, 4, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, 7, None) == DTYPE
    assert h(Q, C, TB, SL, O, 4, 18, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, BF16, None) == SHAPE
    assert h(Q, C, TB, SL, O, -1, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, BF16, None) == SHAPE
    assert h(Q, C, TB, SL, O, 0, 12, 2, 128, 1536, 1536, 64, 16, 8, 0.088, None, BF16, None) == OK


def test_uclip_validation(L):
    f = L.sra_uclip
    X, A, G, O = (P + i * 0x100000 for i in range(4))

    def call(**kw):
        a = dict(x=X, al=A, ga=G, out=O, N=4, H=3, D=64, xn=192, xh=64, on=192, oh=64, apc=1, gpc=0, lo=-1.0,
                 hi=1.0, dt=BF16)
        a.update(kw)
        return f(a["x"], a["al"], a["ga"], a["out"], a["N"], a["H"], a["D"], a["xn"], a["xh"], a["on"], a["oh"],
                 a["apc"], a["gpc"], a["lo"], a["hi"], a["dt"], None)

    assert call(dt=5) == DTYPE
    assert call(N=-1) == SHAPE
    assert call(H=-1) == SHAPE
    assert call(D=0) == SHAPE
    assert call(apc=2) == ARG
    assert call(gpc=-1) == ARG
    assert call(lo=1.0, hi=-1.0) == ARG
    assert call(lo=float("nan")) == ARG
    assert call(hi=float("nan")) == ARG
    assert call(oh=63) == STRIDE                 # heads of out overlap
    assert call(on=100) == STRIDE                # tokens of out overlap
    assert call(xn=-1) == STRIDE
    for name in ("x", "al", "ga", "out"):
        assert call(**{name: None}) == NULL, name
    # heads-outer layout and size-1 dimensions pass the stride check (stopped at NULL)
    assert call(x=None, on=64, oh=256) == NULL
    assert call(x=None, H=1, oh=0, xh=0) == NULL
    assert call(x=None, N=1, on=0, xn=0) == NULL
    assert call(N=0) == OK
    assert call(H=0) == OK
    assert call(out=X + 2) == ALIAS              # x and out overlap, not in place
    assert call(al=O + 4) == ALIAS               # alpha inside out
    assert call(ga=O + 4) == ALIAS


def test_glu_validation(L):
    f = L.sra_glu
    assert f(P, P + 0x100000, 4, 8, 16, 8, 0, 9, None) == DTYPE
    assert f(P, P + 0x100000, 4, 8, 16, 8, 2, BF16, None) == ARG
    assert f(P, P + 0x100000, -1, 8, 16, 8, 0, BF16, None) == SHAPE
    assert f(P, P + 0x100000, 4, 0, 16, 8, 0, BF16, None) == SHAPE
    assert f(P, P + 0x100000, 4, 8, 15, 8, 0, BF16, None) == STRIDE
    assert f(P, P + 0x100000, 4, 8, 16, 7, 0, BF16, None) == STRIDE
    assert f(None, P + 0x100000, 4, 8, 16, 8, 0, BF16, None) == NULL
    assert f(P, P + 8, 4, 8, 16, 8, 0, BF16, None) == ALIAS
    assert f(None, None, 0, 8, 16, 8, 1, BF16, None) == OK
    assert L.sra_swiglu(P, P + 8, 4, 8, 16, 8, BF16, None) == ALIAS


def test_variant_control(L):
    assert sra.variant_count("rmsnorm") == 9
    assert sra.variant_count("rope_kv_store") == 2
    assert sra.variant_count("glu") == 2
    assert [sra.variant_name("glu", i) for i in range(2)] == ["cols_rows", "cols_rows_regs"]
    assert sra.variant_count("linear_narrow") == 1
    assert sra.variant_name("linear_narrow", 0) == "cluster_k_split"
    assert sra.variant_count("decode_attention") == 3
    assert [sra.variant_name("decode_attention", i) for i in range(3)] == ["cuda_cores", "mma_sync", "mma_sync_tma"]
    assert sra.variant_count("linear") == 2
    assert [sra.variant_name("linear", i) for i in range(2)] == ["mma_sync", "tcgen05"]
    assert L.sra_force_variant(b"linear", 1 | (4 << 8)) == OK   # tcgen05 with 4 K splits
    assert L.sra_force_variant(b"linear", 2) == ARG
    assert L.sra_force_variant(b"linear", -1) == OK
    assert sra.variant_count("nope") == ARG
    assert [sra.variant_name("rmsnorm", i) for i in range(9)] == ["warp_rows", "cta_row", "cta_smem", "two_pass",
                                                                  "cta_pair", "warp_smem", "pair_smem", "cta_lean",
                                                                  "warps_row"]
    assert sra.variant_name("rmsnorm", 9) is None
    assert L.sra_force_variant(b"rmsnorm", 9) == ARG
    assert L.sra_force_variant(b"rmsnorm", 8 | (16 << 8) | (4 << 16)) == OK   # warps_row, 16 accesses, 4 warps
    assert L.sra_force_variant(b"rmsnorm", 1 | (2 << 24)) == OK   # cta_row, at most 2 CTAs per SM
    assert L.sra_force_variant(b"rmsnorm", 1 << 28) == ARG
    assert L.sra_force_variant(b"bogus", 0) == ARG
    assert L.sra_force_variant(b"rmsnorm", 2) == OK
    assert sra.pick_variant("rmsnorm", 512, 1536, num_sms=152) == 2
    assert L.sra_force_variant(b"rmsnorm", -1) == OK


def test_dispatch_choices(L):
    import torch

    pick = sra.pick_variant
    # short rows, many of them: one warp per row
    assert pick("rmsnorm", 4096, 1536, dtype=torch.bfloat16, num_sms=152) == 0
    # decode (few rows) of the 1536-wide hidden state: a CTA per row
    assert pick("rmsnorm", 1, 1536, dtype=torch.bfloat16, num_sms=152) == 1
    assert pick("rmsnorm", 64, 1536, dtype=torch.bfloat16, num_sms=152) == 1
    # from 256 rows of 1536: one warp per row (measured 15 % faster at 256 rows)
    assert pick("rmsnorm", 256, 1536, dtype=torch.bfloat16, num_sms=152) == 0
    # rows of 257 to 512 16-byte accesses, a few hundred of them: a warp per row (12 or 16
    # accesses per lane); more rows keep the CTA variants
    assert pick("rmsnorm", 512, 4096, dtype=torch.bfloat16, num_sms=152) == 0
    assert pick("rmsnorm", 512, 2176, dtype=torch.bfloat16, num_sms=152) == 0
    assert pick("rmsnorm", 512, 1536, dtype=torch.float32, num_sms=152) == 0
    assert pick("rmsnorm", 512, 2048, dtype=torch.float32, num_sms=152) == 0
    assert pick("rmsnorm", 4096, 4096, dtype=torch.bfloat16, num_sms=152) == 7
    # 16-bit rows of 8192 elements, 512 of them: the lean CTA per row
    assert pick("rmsnorm", 512, 8192, dtype=torch.float16, num_sms=152) == 7
    # a row past a warp's registers: CTA per row
    assert pick("rmsnorm", 512, 2176, dtype=torch.float32, num_sms=152) == 1
    # wide rows, 512 of them on 152 SMs: a CTA per row (measured faster than a CTA pair)
    assert pick("rmsnorm", 512, 8192, dtype=torch.float32, num_sms=152) == 1
    # past a CTA's registers: the row landed in shared memory
    assert pick("rmsnorm", 64, 40000, dtype=torch.bfloat16, num_sms=152) == 2
    # past shared memory: two-pass
    assert pick("rmsnorm", 2, 10_000_000, dtype=torch.float32, num_sms=152) == 3
    # SiLU with the registers the compiler picks, ReLU held to 48 (measured)
    assert pick("glu", 4096, 14336, num_sms=152) == 1
    assert pick("glu", 4096, 14336, 1, num_sms=152) == 0
    # RoPE: one task per thread up to 8 tokens per SM, two tasks per thread past that (an even
    # number of head units); an odd number keeps one task per thread
    assert pick("rope_kv_store", 64, 12, 2, 128, num_sms=152) == 0
    assert pick("rope_kv_store", 1216, 12, 2, 128, num_sms=152) == 0
    assert pick("rope_kv_store", 2048, 12, 2, 128, num_sms=152) == 1
    assert pick("rope_kv_store", 2048, 3, 1, 64, num_sms=152) == 0
    # the threshold follows the SM count: past 8 tokens per SM
    assert pick("rope_kv_store", 800, 12, 2, 128, num_sms=100) == 0
    assert pick("rope_kv_store", 801, 12, 2, 128, num_sms=100) == 1
    # warp rows of 257-512 accesses only between 256 rows and 8 rows per SM
    assert pick("rmsnorm", 255, 1536, dtype=torch.float32, num_sms=152) == 1
    assert pick("rmsnorm", 256, 1536, dtype=torch.float32, num_sms=152) == 0
    assert pick("rmsnorm", 1216, 1536, dtype=torch.float32, num_sms=152) == 0
    assert pick("rmsnorm", 1217, 1536, dtype=torch.float32, num_sms=152) == 1
    # past 512 accesses (fp32 2176: 544) a warp cannot hold the row
    assert pick("rmsnorm", 512, 2176, dtype=torch.float32, num_sms=152) == 1
    # decode attention: tensor cores for 16-bit data up to head_dim 128, CUDA cores otherwise
    assert pick("decode_attention", 32, 12, 2, 128, dtype=torch.bfloat16, num_sms=152) == 1
    assert pick("decode_attention", 32, 12, 2, 256, dtype=torch.bfloat16, num_sms=152) == 0
    assert pick("decode_attention", 32, 12, 2, 128, dtype=torch.float32, num_sms=152) == 0
    assert pick("decode_attention", 32, 18, 2, 128, num_sms=152) == SHAPE
    assert pick("rmsnorm", -1, 16, num_sms=152) == SHAPE


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="would launch on fake pointers")
def test_interleaved_views_are_not_aliases(L):
    """q / k / v as interleaved views of one fused QKV buffer pass the alias check
    (the call then stops at the device query on this GPU-less host)."""
    DEVICE = -9
    T, nh, nkv, hd = 8, 12, 2, 128
    W = (nh + 2 * nkv) * hd   # token stride of the fused buffer, elements
    base = 0x100000
    q, k, v = base, base + nh * hd * 2, base + (nh + nkv) * hd * 2
    cache = 0x10000000
    args = lambda q_, k_, v_: (q_, k_, v_, 0x2000000, 0x3000000, 0x4000000, 0x5000000, cache, T, nh, nkv, hd,
                                W, W, W, 32768, 16, 16, None, BF16, None)
    assert L.sra_rope_kv_store(*args(q, k, v)) == DEVICE
    # k starting inside q's row of the same token: a real overlap
    assert L.sra_rope_kv_store(*args(q, q + 64, v)) == ALIAS
    # gate_up and out interleaved in one buffer of stride 3I: disjoint
    I = 64
    assert L.sra_glu(base, base + 2 * I * 2, 4, I, 3 * I, 3 * I, 0, BF16, None) == DEVICE
    assert L.sra_glu(base, base + I * 2, 4, I, 3 * I, 3 * I, 0, BF16, None) == ALIAS
    # uclip in place on the K heads of a fused QKV buffer
    assert L.sra_uclip(k, 0x2000000, 0x3000000, k, T, nkv, hd, W, hd, W, hd, 1, 1, -1.0, 1.0, BF16, None) == DEVICE
    # uclip from the Q heads into the K heads of the same buffer: disjoint
    assert L.sra_uclip(q, 0x2000000, 0x3000000, k, T, nkv, hd, W, hd, W, hd, 1, 1, -1.0, 1.0, BF16, None) == DEVICE
    # add_rmsnorm: x | res | out interleaved rows of one [rows, 3D] buffer
    D = 32
    assert L.sra_add_rmsnorm(base, base + D * 2, 0x900000, base + 2 * D * 2, 4, D, 3 * D, 3 * D, 3 * D, 1e-6,
                             BF16, None) == DEVICE
