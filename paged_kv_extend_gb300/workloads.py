"""Seeded synthetic workloads for extend / decode attention over a paged pool.

This module only draws inputs: lengths, slot assignments, index arrays and
bf16 values.  It holds none of the attention arithmetic, imports nothing from
the CUDA library or the oracle, and is the one module both of them are fed
from.

Recipe (the same for every workload):
  * a CPU ``torch.Generator`` seeded with ``seed`` draws, in this order, the
    per-sequence prefix/extend lengths, a random permutation of the pool's
    slots, then K rows, V rows and Q rows;
  * sequence b's T_b = P_b + E_b tokens take the next T_b entries of the slot
    permutation: the first P_b are its cached prefix, the last E_b its new
    (extend) tokens;
  * K/V of every token are written into the pool at its slot; the extend
    tokens' K/V are also handed out contiguously (``k_extend``/``v_extend``),
    as a serving engine holds them right after the QKV projection;
  * values are bf16 draws from N(0, std^2).
  * MLA workloads (Lq=576, Lv=512) store one latent row per token; V is a
    view of its first 512 dims, as in sglang's MLA layout.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


@dataclasses.dataclass
class WorkloadSpec:
    """Shape of one workload.  Lengths are either a list (one entry per
    sequence) or a distribution tuple: ("uniform", lo, hi) inclusive,
    ("const", n), ("lognormal", mu, sigma, lo, hi) rounded and clipped."""
    name: str
    batch: int
    hq: int
    hkv: int
    lq: int
    lv: int
    prefix: object
    extend: object
    num_slots: int
    sm_scale: float = 0.0          # <= 0: 1/sqrt(lq)
    logit_cap: float = 0.0         # <= 0: off
    sliding_window: int = -1       # <= 0: off
    std: float = 1.0
    seed: int = 1000
    v_aliases_k: bool = False      # MLA: V = first lv dims of K
    decode: bool = False           # one query per sequence over all T_b keys
    tree_mask: bool = False        # custom mask: each extend token is a draft-tree
                                   # node that sees the prefix, its ancestors and itself
    sinks: bool = False            # a sink logit per query head

    @property
    def group(self) -> int:
        return self.hq // self.hkv


# Workloads shaped like the pages' (GQA Llama/Qwen-style heads, MLA 576/512,
# ragged prefix/extend mixes).  Seeds are 1000 + the workload's index.
SPECS = {
    "tiny": WorkloadSpec(
        "tiny", batch=2, hq=4, hkv=2, lq=64, lv=64, prefix=[16, 0],
        extend=[8, 5], num_slots=64, sm_scale=1.0 / 8.0, seed=1000),
    "llama3_8b": WorkloadSpec(
        "llama3_8b", batch=16, hq=32, hkv=8, lq=128, lv=128,
        prefix=("uniform", 0, 4096), extend=("uniform", 1, 1024),
        num_slots=262144, sm_scale=1.0 / math.sqrt(128.0), seed=1001),
    "long_prefix": WorkloadSpec(
        "long_prefix", batch=64, hq=32, hkv=8, lq=128, lv=128,
        prefix=("const", 8192), extend=("const", 16), num_slots=1 << 20,
        logit_cap=30.0, seed=1002),
    "mla": WorkloadSpec(
        "mla", batch=8, hq=16, hkv=1, lq=576, lv=512, prefix=("const", 2048),
        extend=("const", 512), num_slots=65536, sm_scale=1.0 / math.sqrt(192.0),
        std=0.5, seed=1003, v_aliases_k=True),
    "heavy_tail": WorkloadSpec(
        "heavy_tail", batch=256, hq=28, hkv=4, lq=128, lv=128,
        prefix=("lognormal", 6.0, 1.2, 0, 16384),
        extend=("lognormal", 6.0, 1.2, 1, 4096), num_slots=1 << 22,
        sliding_window=4096, seed=1004),
    # Decode shapes derived from the long-prefix and MLA workloads: one query
    # per sequence over T keys, the current token's K/V already in the pool.
    "decode_gqa": WorkloadSpec(
        "decode_gqa", batch=64, hq=32, hkv=8, lq=128, lv=128,
        prefix=("const", 8192), extend=("const", 1), num_slots=1 << 20,
        seed=1005, decode=True),
    "decode_mla": WorkloadSpec(
        "decode_mla", batch=64, hq=16, hkv=1, lq=576, lv=512,
        prefix=("const", 4095), extend=("const", 1), num_slots=1 << 20,
        sm_scale=1.0 / math.sqrt(192.0), std=0.5, seed=1006, v_aliases_k=True,
        decode=True),
    # Speculative-decoding verification: a 64-node draft tree per sequence
    # over its cached prefix, under a custom (tree) mask.
    "spec_verify": WorkloadSpec(
        "spec_verify", batch=64, hq=32, hkv=8, lq=128, lv=128,
        prefix=("uniform", 1024, 4096), extend=("const", 64), num_slots=1 << 20,
        seed=1007, tree_mask=True),
    # A layer with attention sinks and a 128-token sliding window (64-dim
    # heads, 64 query / 8 KV heads).
    "sinks_swa": WorkloadSpec(
        "sinks_swa", batch=16, hq=64, hkv=8, lq=64, lv=64,
        prefix=("uniform", 0, 4096), extend=("uniform", 1, 1024), num_slots=1 << 18,
        sliding_window=128, seed=1008, sinks=True),
    # The split head dims of the pages' launcher (Lq = 192 = 128 + 64 rope with
    # Lv = 128, and Lq = 288 = 256 + 32 rope with Lv = 256) on the
    # Llama-shaped length mix; 16 query heads each, one KV head per query head
    # for 192 / 128 (an MHA latent-free layout) and groups of four for 288.
    "split_192": WorkloadSpec(
        "split_192", batch=16, hq=16, hkv=16, lq=192, lv=128,
        prefix=("uniform", 0, 4096), extend=("uniform", 1, 1024), num_slots=1 << 18,
        sm_scale=1.0 / math.sqrt(192.0), seed=1009),
    "split_288": WorkloadSpec(
        "split_288", batch=16, hq=16, hkv=4, lq=288, lv=256,
        prefix=("uniform", 0, 4096), extend=("uniform", 1, 1024), num_slots=1 << 18,
        sm_scale=1.0 / math.sqrt(288.0), seed=1010),
}


def _draw_lengths(dist, n: int, g: torch.Generator) -> List[int]:
    if isinstance(dist, (list, tuple)) and (len(dist) == 0 or not isinstance(dist[0], str)):
        assert len(dist) == n
        return [int(x) for x in dist]
    kind = dist[0]
    if kind == "const":
        return [int(dist[1])] * n
    if kind == "uniform":
        lo, hi = int(dist[1]), int(dist[2])
        return torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    if kind == "lognormal":
        mu, sigma, lo, hi = float(dist[1]), float(dist[2]), int(dist[3]), int(dist[4])
        z = torch.randn(n, generator=g, dtype=torch.float64)
        vals = torch.exp(mu + sigma * z).round().clamp(lo, hi)
        return [int(x) for x in vals.tolist()]
    raise ValueError(f"unknown length distribution {dist!r}")


def _cumsum0(lens: List[int]) -> torch.Tensor:
    out = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if lens:
        out[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return out


def _bf16_normal(shape, std: float, g: torch.Generator) -> torch.Tensor:
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


@dataclasses.dataclass
class Workload:
    """CPU tensors of one drawn workload.

    Per-token rows are stored compactly (``k_rows``/``v_rows`` indexed by the
    token's position in the batch's concatenated [prefix_b, extend_b] order);
    :meth:`pool` scatters them into a full [num_slots, Hkv, D] pool.
    """
    spec: WorkloadSpec
    prefix_lens: List[int]
    extend_lens: List[int]
    slots: torch.Tensor            # int32 [sum T]  slot of each token
    k_rows: torch.Tensor           # bf16 [sum T, Hkv, Lq]
    v_rows: torch.Tensor           # bf16 [sum T, Hkv, Lv] (view of k_rows for MLA)
    q: torch.Tensor                # bf16 [sum E, Hq, Lq]  (decode: [B, Hq, Lq])
    qo_indptr: torch.Tensor        # int32 [B+1] cumsum of E
    kv_indptr: torch.Tensor        # int32 [B+1] cumsum of P (decode: of T)
    kv_indices: torch.Tensor       # int32 [sum P] prefix slots (decode: all slots)
    extend_kv_indices: torch.Tensor  # int32 [sum E] slots of the extend tokens
    extend_start_loc: torch.Tensor   # int32 [B]
    extend_seq_lens: torch.Tensor    # int32 [B]
    token_offsets: torch.Tensor      # int64 [B+1] start of sequence b in k_rows
    custom_mask: Optional[torch.Tensor] = None  # uint8, row i of b at mask_indptr[b] + i*T_b
    mask_indptr: Optional[torch.Tensor] = None  # int32 [B+1]
    sinks: Optional[torch.Tensor] = None        # fp32 [Hq]

    @property
    def batch(self) -> int:
        return self.spec.batch

    @property
    def n_q_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def sm_scale(self) -> float:
        s = self.spec.sm_scale
        return s if s and s > 0 else 1.0 / math.sqrt(self.spec.lq)

    def extend_rows(self) -> torch.Tensor:
        """Indices into k_rows/v_rows of the extend tokens, in qo order."""
        idx = []
        for b in range(self.batch):
            t0 = int(self.token_offsets[b]) + self.prefix_lens[b]
            idx.append(torch.arange(t0, t0 + self.extend_lens[b], dtype=torch.int64))
        return torch.cat(idx) if idx else torch.zeros(0, dtype=torch.int64)

    def extend_kv(self, device="cpu"):
        """(k_extend [sum E, Hkv, Lq], v_extend [sum E, Hkv, Lv]) on device."""
        rows = self.extend_rows()
        k = self.k_rows.index_select(0, rows).to(device)
        if self.spec.v_aliases_k:
            return k, k[..., : self.spec.lv]
        return k, self.v_rows.index_select(0, rows).to(device)

    def pool_fp8(self, dtype, k_scale: float, v_scale: float, device="cpu"):
        """The pool in an fp8 format (torch.float8_e4m3fn or float8_e5m2):
        every token row divided by its scale and converted by torch, zero
        elsewhere.  (k_buffer, v_buffer) as one-byte tensors of that dtype; for
        MLA, v_buffer is a view of k_buffer."""
        s = self.spec
        slots = self.slots.to(torch.int64)
        k = torch.zeros(s.num_slots, s.hkv, s.lq, dtype=torch.uint8)
        if slots.numel():
            k[slots] = (self.k_rows.float() / k_scale).to(dtype).view(torch.uint8)
        if s.v_aliases_k:
            # MLA: v_buffer is a view of the first Lv codes of k_buffer (a
            # value reads code * v_scale)
            kd = k.view(dtype).to(device)
            return kd, kd[..., : s.lv]
        v = torch.zeros(s.num_slots, s.hkv, s.lv, dtype=torch.uint8)
        if slots.numel():
            v[slots] = (self.v_rows.float() / v_scale).to(dtype).view(torch.uint8)
        return k.view(dtype).to(device), v.view(dtype).to(device)

    def req_to_token(self, rows: Optional[int] = None, cols: Optional[int] = None,
                     seed: int = 0):
        """A request-to-token table holding this batch: sequence b sits in a
        random row req_pool_indices[b] (row 0 stays reserved and all zero),
        its T_b slots in columns [0, T_b) in key order; every other entry is a
        random slot.  Returns (req_to_token int32 [rows, cols],
        req_pool_indices int64 [B], seq_lens int64 [B])."""
        g = torch.Generator().manual_seed(seed)
        t = [p + e for p, e in zip(self.prefix_lens, self.extend_lens)]
        rows = rows if rows is not None else 2 * self.batch + 1
        cols = cols if cols is not None else max(t + [1]) + 7
        table = torch.randint(0, max(self.spec.num_slots, 1), (rows, cols),
                              generator=g, dtype=torch.int32)
        table[0] = 0
        rpi = (torch.randperm(rows - 1, generator=g)[: self.batch] + 1).to(torch.int64)
        for b in range(self.batch):
            o = int(self.token_offsets[b])
            table[int(rpi[b]), : t[b]] = self.slots[o: o + t[b]]
        return table, rpi, torch.tensor(t, dtype=torch.int64)

    def pool(self, device="cpu"):
        """(k_buffer [S, Hkv, Lq], v_buffer [S, Hkv, Lv]) on device, zero
        except at the workload's slots.  For MLA, v_buffer is a view of the
        first Lv dims of k_buffer."""
        s = self.spec
        slots = self.slots.to(device=device, dtype=torch.int64)
        k = torch.zeros(s.num_slots, s.hkv, s.lq, dtype=torch.bfloat16, device=device)
        if slots.numel():
            k.index_copy_(0, slots, self.k_rows.to(device))
        if s.v_aliases_k:
            return k, k[..., : s.lv]
        v = torch.zeros(s.num_slots, s.hkv, s.lv, dtype=torch.bfloat16, device=device)
        if slots.numel():
            v.index_copy_(0, slots, self.v_rows.to(device))
        return k, v


def draw(spec: WorkloadSpec, seed: Optional[int] = None) -> Workload:
    """Draw one workload from ``spec`` (seed defaults to ``spec.seed``)."""
    g = torch.Generator().manual_seed(spec.seed if seed is None else seed)
    b = spec.batch
    if spec.decode:
        # decode: T_b = prefix + the current token, all in the pool
        p = _draw_lengths(spec.prefix, b, g)
        e = _draw_lengths(spec.extend, b, g)
    else:
        p = _draw_lengths(spec.prefix, b, g)
        e = _draw_lengths(spec.extend, b, g)
    t = [pi + ei for pi, ei in zip(p, e)]
    total = sum(t)
    if total > spec.num_slots:
        raise ValueError(f"{spec.name}: {total} tokens do not fit {spec.num_slots} slots")
    perm = torch.randperm(spec.num_slots, generator=g)[:total].to(torch.int32)
    k_rows = _bf16_normal((total, spec.hkv, spec.lq), spec.std, g)
    if spec.v_aliases_k:
        v_rows = k_rows[..., : spec.lv]
    else:
        v_rows = _bf16_normal((total, spec.hkv, spec.lv), spec.std, g)
    n_q = b if spec.decode else sum(e)
    q = _bf16_normal((n_q, spec.hq, spec.lq), spec.std, g)

    offs = [0]
    for ti in t:
        offs.append(offs[-1] + ti)
    pre_idx, ext_idx = [], []
    for i in range(b):
        pre_idx.append(perm[offs[i]: offs[i] + p[i]])
        ext_idx.append(perm[offs[i] + p[i]: offs[i + 1]])
    cat = lambda xs: torch.cat(xs) if xs else torch.zeros(0, dtype=torch.int32)
    if spec.decode:
        kv_indptr = _cumsum0(t)
        kv_indices = perm.clone()
        qo_indptr = _cumsum0([1] * b)
    else:
        kv_indptr = _cumsum0(p)
        kv_indices = cat(pre_idx)
        qo_indptr = _cumsum0(e)
    # drawn after everything else, so the other fields do not depend on them
    custom_mask = mask_indptr = sinks = None
    if spec.tree_mask and not spec.decode:
        rows, mptr = [], [0]
        for i in range(b):
            E, P = e[i], p[i]
            anc = torch.zeros(E, E, dtype=torch.bool)     # anc[n, a]: a is n or an ancestor
            for n in range(E):
                if n > 0:
                    parent = int(torch.randint(0, n, (1,), generator=g))
                    anc[n] = anc[parent]
                anc[n, n] = True
            m = torch.cat([torch.ones(E, P, dtype=torch.bool), anc], dim=1)
            rows.append(m.to(torch.uint8).reshape(-1))
            mptr.append(mptr[-1] + E * (P + E))
        custom_mask = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.uint8)
        mask_indptr = torch.tensor(mptr, dtype=torch.int32)
    if spec.sinks:
        sinks = torch.randn(spec.hq, generator=g) * 1.5
    return Workload(
        spec=spec, prefix_lens=p, extend_lens=e, slots=perm, k_rows=k_rows,
        v_rows=v_rows, q=q, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
        kv_indices=kv_indices.to(torch.int32), extend_kv_indices=cat(ext_idx).to(torch.int32),
        extend_start_loc=_cumsum0(e)[:-1].clone(),
        extend_seq_lens=torch.tensor(e, dtype=torch.int32),
        token_offsets=torch.tensor(offs, dtype=torch.int64),
        custom_mask=custom_mask, mask_indptr=mask_indptr, sinks=sinks)


def small_spec(name="rand", batch=3, hq=8, hkv=2, lq=128, lv=128, prefix=None,
               extend=None, num_slots=None, seed=7, **kw) -> WorkloadSpec:
    """A small ragged workload for tests: explicit per-sequence lengths, a
    pool just large enough (x2) for every token."""
    prefix = prefix if prefix is not None else [5, 0, 130][:batch]
    extend = extend if extend is not None else [3, 17, 200][:batch]
    total = sum(prefix) + sum(extend)
    if num_slots is None:
        num_slots = max(16, 2 * total)
    return WorkloadSpec(name, batch=batch, hq=hq, hkv=hkv, lq=lq, lv=lv,
                        prefix=list(prefix), extend=list(extend),
                        num_slots=num_slots, seed=seed, **kw)
