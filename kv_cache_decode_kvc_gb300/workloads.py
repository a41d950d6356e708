"""The decode workloads the pages describe, as shapes (no arithmetic).

T is the number of tokens already cached before the step; the step appends one more, so
every sequence attends over L_b = T_b + 1 slots and T_max = max_b L_b.  Values are bf16
draws of the counter-based generator in :mod:`synth` (the pages name no dataset).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import synth


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    B: int
    H_q: int
    H_kv: int
    D: int
    T: int | None          # uniform cached length, or None for the ragged range below
    T_lo: int = 0
    T_hi: int = 0
    dtype: str = "bf16"
    seed: int = 1234
    note: str = ""

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def lens_pre(self) -> torch.Tensor:
        """Cached length of each sequence before the step (int32, CPU)."""
        if self.T is not None:
            return torch.full((self.B,), self.T, dtype=torch.int32)
        return synth.uniform_lens(self.seed, self.B, self.T_lo, self.T_hi)

    def lens(self) -> torch.Tensor:
        return self.lens_pre() + 1

    def T_max(self) -> int:
        return int(self.lens().max())

    def kv_read_bytes_per_layer(self, window: int = 0, new_tokens: int = 1, int8: bool = False) -> int:
        """Algorithmic KV bytes one decode step reads per layer: 2 H_kv D s sum_b L_b, with
        L_b capped at the window for sliding-window attention (window > 0), and L_b = T_b +
        new_tokens when a step appends several tokens (the keys are read once for all of them).
        An int8 cache reads D one-byte codes and one 4-byte scale per row instead of D s."""
        lens = self.lens_pre() + new_tokens
        if window > 0:
            lens = lens.clamp(max=window)
        row = self.D + 4 if int8 else self.D * self.elem_bytes
        return 2 * self.H_kv * row * int(lens.sum())


WORKLOADS = {
    w.name: w
    for w in [
        Workload("llama2_7b_mha_b1_t4096", 32, 1, 32, 32, 128, 4096,
                 note="Llama-2-7B-shaped MHA, every sequence at 4096 cached tokens"),
        Workload("gqa8b_b24_ragged3000_6000", 32, 24, 32, 8, 128, None, 3000, 6000,
                 note="8B-shaped GQA serving batch, cached lengths U{3000..6000} (seed 1234)"),
        Workload("gqa70b_b32_t8192", 80, 32, 64, 8, 128, 8192,
                 note="70B-shaped GQA long context (80 GiB cache)"),
        # the MQA shapes are single-layer; 4 layer copies make a step read 4x their bytes, more
        # than L2 holds, so that timed reads come from HBM
        Workload("mqa_b64_t4096", 4, 64, 32, 1, 128, 4096, note="MQA, one layer's shape x 4 copies"),
        Workload("mqa_b1_t131072", 4, 1, 32, 1, 128, 131072,
                 note="MQA long context, split-T stress, one layer's shape x 4 copies"),
    ]
}

HEADLINE = "gqa8b_b24_ragged3000_6000"


def paged_table(w: Workload, block_size: int, spare: int = 0):
    """Block table for a paged copy of the workload: every sequence gets ceil(T_max / block_size)
    logical blocks, mapped to a seeded random permutation of a pool with `spare` unused blocks,
    so logically adjacent blocks are never adjacent in memory.  Returns (table int32 [B,
    max_blocks] on the CPU, num_blocks, max_blocks)."""
    max_blocks = -(-w.T_max() // block_size)
    num_blocks = w.B * max_blocks + spare
    g = torch.Generator().manual_seed(w.seed + 101 * block_size)
    table = torch.randperm(num_blocks, generator=g)[: w.B * max_blocks].to(torch.int32)
    return table.view(w.B, max_blocks).contiguous(), num_blocks, max_blocks


def fill_layer(cache, layer: int, w: Workload, seed: int | None = None, device="cuda",
               chunk_elems: int = 1 << 26, table=None):
    """Write the layer's seeded history (slots [0, T_b)) through kvc_prefill_write (through
    kvc_paged_prefill_write with `table`, a device block table, for a paged cache)."""
    seed = w.seed if seed is None else seed
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    lp = w.lens_pre()
    T_in = int(lp.max())
    per_b = w.H_kv * T_in * w.D
    step = max(1, chunk_elems // per_b)
    K = torch.empty(w.B, w.H_kv, T_in, w.D, dtype=dt, device=device)
    V = torch.empty_like(K)
    for b0 in range(0, w.B, step):
        b1 = min(w.B, b0 + step)
        K[b0:b1] = synth.block(seed, layer, "K", b0, b1, w.H_kv, 0, T_in, w.D, w.B, dt, device)
        V[b0:b1] = synth.block(seed, layer, "V", b0, b1, w.H_kv, 0, T_in, w.D, w.B, dt, device)
    if table is None:
        cache.prefill_write(layer, K, V, lp.to(device))
    else:
        cache.prefill_write(layer, K, V, table, lp.to(device))
    del K, V


def step_inputs(w: Workload, layer: int, seed: int | None = None, device="cuda"):
    """q [B,H_q,D], k_new / v_new [B,H_kv,D] (the generator's row T_b of each stream)."""
    seed = w.seed if seed is None else seed
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    lp = w.lens_pre()
    q = synth.queries(seed, layer, w.B, w.H_q, w.D, dt, device)
    # row T_b of stream (b, h): gather with one generator call per distinct length
    kn = torch.empty(w.B, w.H_kv, w.D, dtype=dt, device=device)
    vn = torch.empty_like(kn)
    for T_b in sorted(set(lp.tolist())):
        idx = [b for b in range(w.B) if int(lp[b]) == T_b]
        for b in idx:
            kn[b] = synth.block(seed, layer, "K", b, b + 1, w.H_kv, T_b, T_b + 1, w.D, w.B, dt, device)[0, :, 0]
            vn[b] = synth.block(seed, layer, "V", b, b + 1, w.H_kv, T_b, T_b + 1, w.D, w.B, dt, device)[0, :, 0]
    return q, kn, vn


def step_inputs_multi(w: Workload, layer: int, T_q: int, seed: int | None = None, device="cuda"):
    """A step with T_q new tokens per sequence: q [B,H_q,T_q,D] (rows 0..T_q-1 of tensor 'Q'),
    k_new / v_new [B,H_kv,T_q,D] (the generator's rows T_b .. T_b + T_q - 1 of each stream)."""
    seed = w.seed if seed is None else seed
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    lp = w.lens_pre()
    q = synth.block(seed, layer, "Q", 0, w.B, w.H_q, 0, T_q, w.D, w.B, dt, device).contiguous()
    kn = torch.empty(w.B, w.H_kv, T_q, w.D, dtype=dt, device=device)
    vn = torch.empty_like(kn)
    for b in range(w.B):
        t0 = int(lp[b])
        kn[b] = synth.block(seed, layer, "K", b, b + 1, w.H_kv, t0, t0 + T_q, w.D, w.B, dt, device)[0]
        vn[b] = synth.block(seed, layer, "V", b, b + 1, w.H_kv, t0, t0 + T_q, w.D, w.B, dt, device)[0]
    return q, kn, vn
