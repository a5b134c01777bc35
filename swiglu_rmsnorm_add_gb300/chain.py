"""The per-token decoder-layer chain: add_rmsnorm -> rope_kv_store -> add_rmsnorm
-> swiglu, repeated over the layers, at decode batch B.

This is the bandwidth-bound part of one decode step of a Qwen2.5-1.5B-shaped
model (koas-w.github.io "preformanceimprovement": 28 layers, 2 norms per
layer, the fused RoPE/KV store and SwiGLU; m.lsln.cn/news/61269 section 4:
launch overhead per kernel and CUDA-graph replay of the whole step). The dense
projections between these kernels (QKV, attention, o_proj, gate_up, down) are
not part of this path: their outputs are seeded activations held in static
buffers, as a CUDA graph needs (same page, section 4.2).

Per layer l:
    x  <- x + attn_res[l];  h1[l]  = rmsnorm(x) * w_ln1[l]
    rope_kv_store(q[l], k[l], v[l], cos, sin, pos, slots[l], kv_cache[l])
    x  <- x + mlp_res[l];   h2[l]  = rmsnorm(x) * w_ln2[l]
    act[l] = silu(gate_up[l][:, :I]) * gate_up[l][:, I:]
Every call goes through the C ABI; there are 4 * layers launches per step.
"""
from __future__ import annotations

import torch

from . import _binding as sra
from . import synthetic as syn


class DecodeChain:
    def __init__(self, batch: int, layers: int = 28, hidden: int = 1536, n_head: int = 12, n_kv_head: int = 2,
                 head_dim: int = 128, intermediate: int = 8960, num_blocks: int = 4096, block_size: int = 16,
                 max_pos: int = 32768, theta: float = 1e6, seed: int = 1004, device="cuda",
                 dtype=torch.bfloat16):
        self.B, self.L, self.H, self.I = batch, layers, hidden, intermediate
        self.n_head, self.n_kv, self.hd = n_head, n_kv_head, head_dim
        self.num_blocks, self.block_size = num_blocks, block_size
        self.eps = syn.EPS
        self.dtype = dtype
        dev = torch.device(device)
        B = batch

        def n(shape, mean, std, stream):
            return syn.normal(shape, mean, std, dtype, seed, stream).to(dev)

        cos, sin = syn.rope_tables(max_pos, head_dim, theta)
        self.cos, self.sin = cos.to(dev), sin.to(dev)
        self.pos = syn.positions(B, max_pos, seed, 1).to(dev)
        self.x = n((B, hidden), 0.0, 1.0, 2)
        self.layers = []
        for l in range(layers):
            s = 100 + 20 * l
            lay = dict(
                attn_res=n((B, hidden), 0.0, 1.0, s + 1),
                w_ln1=n((hidden,), 1.0, 0.1, s + 2),
                q=n((B, n_head, head_dim), 0.0, 1.0, s + 3),
                k=n((B, n_kv_head, head_dim), 0.0, 1.0, s + 4),
                v=n((B, n_kv_head, head_dim), 0.0, 1.0, s + 5),
                slots=syn.slots(B, num_blocks * block_size, seed, s + 6).to(dev),
                kv_cache=syn.sentinel_cache((2, num_blocks, block_size, n_kv_head, head_dim), dtype).to(dev),
                mlp_res=n((B, hidden), 0.0, 1.0, s + 7),
                w_ln2=n((hidden,), 1.0, 0.1, s + 8),
                gate_up=n((B, 2 * intermediate), 0.0, 1.0, s + 9),
                h1=torch.empty(B, hidden, dtype=dtype, device=dev),
                h2=torch.empty(B, hidden, dtype=dtype, device=dev),
                act=torch.empty(B, intermediate, dtype=dtype, device=dev),
            )
            self.layers.append(lay)
        self.graph = None

    # ------------------------------------------------------------ one layer
    def layer_calls(self, l: int):
        """The layer's four calls as (name, thunk) pairs, in chain order."""
        L = self.layers[l]
        return [
            ("add_rmsnorm", lambda: sra.add_rmsnorm(self.x, L["attn_res"], L["w_ln1"], L["h1"], self.eps)),
            ("rope_kv_store", lambda: sra.rope_kv_store(L["q"], L["k"], L["v"], self.cos, self.sin, self.pos,
                                                        L["slots"], L["kv_cache"])),
            ("add_rmsnorm", lambda: sra.add_rmsnorm(self.x, L["mlp_res"], L["w_ln2"], L["h2"], self.eps)),
            ("swiglu", lambda: sra.swiglu(L["gate_up"], L["act"])),
        ]

    def step(self) -> None:
        """One token step, launched eagerly (4 * layers launches)."""
        for l in range(self.L):
            for _, call in self.layer_calls(l):
                call()

    def capture(self, pdl: bool = True, warmup: bool = True) -> torch.cuda.CUDAGraph:
        """Capture one step into a CUDA graph (after one eager warm-up step unless
        warmup=False). With pdl, each launch is captured with programmatic
        stream serialization, so a kernel's launch overlaps the tail of the one
        before it."""
        prev = sra.set_pdl(pdl)
        try:
            if warmup:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    self.step()
                torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step()
        finally:
            sra.set_pdl(prev)
        self.graph = g
        return g

    def replay(self) -> None:
        self.graph.replay()

    def capture_kind(self, kind: str, pdl: bool = True) -> torch.cuda.CUDAGraph:
        """A CUDA graph of only the step's calls of one kernel kind ("add_rmsnorm",
        "rope_kv_store" or "swiglu"), in chain order on the chain's own buffers: the
        per-launch time of that kind inside a dependent chain, for per-kernel
        accounting of the step."""
        prev = sra.set_pdl(pdl)
        try:
            calls = [c for l in range(self.L) for k, c in self.layer_calls(l) if k == kind]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in calls:
                    c()
        finally:
            sra.set_pdl(prev)
        return g

    def launches_per_step(self) -> dict:
        return {"add_rmsnorm": 2 * self.L, "rope_kv_store": self.L, "swiglu": self.L}

    # ------------------------------------------------------------ accounting
    def bytes_per_step(self) -> dict:
        """Algorithmic HBM bytes of one step, per kernel kind (weights counted once)."""
        s = torch.tensor([], dtype=self.dtype).element_size()
        B, H, I, L = self.B, self.H, self.I, self.L
        nh, nkv, hd = self.n_head, self.n_kv, self.hd
        addn = 4 * B * H * s + H * s
        rope = B * (2 * nh * hd * s + 2 * nkv * hd * s + 2 * (hd // 2) * 4 + 8 + 8 + 2 * nkv * hd * s)
        glu = B * (2 * I * s + I * s)
        return {"add_rmsnorm": 2 * L * addn, "rope_kv_store": L * rope, "swiglu": L * glu}
