"""Helpers shared by the GPU parity tests: run the CUDA path (through the C
ABI) and the float64 oracle on the same seeded workload, and compare."""
import torch

import oracle
from paged_kv_extend_gb300 import pkx
from paged_kv_extend_gb300 import workloads as W

# Tolerances for bf16 outputs against the float64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 1e-3

DEV = torch.device("cuda:0")


class DeviceWorkload:
    """A workload's tensors on the GPU (pool, extend K/V, q, indices)."""

    def __init__(self, wl: W.Workload):
        self.wl = wl
        s = wl.spec
        self.k_buffer, self.v_buffer = wl.pool(DEV)
        self.q = wl.q.to(DEV)
        self.qo_indptr = wl.qo_indptr.to(DEV)
        self.kv_indptr = wl.kv_indptr.to(DEV)
        self.kv_indices = wl.kv_indices.to(DEV)
        if not s.decode:
            self.k_extend, self.v_extend = wl.extend_kv(DEV)
            self.extend_kv_indices = wl.extend_kv_indices.to(DEV)
            self.extend_start_loc = wl.extend_start_loc.to(DEV)
            self.extend_seq_lens = wl.extend_seq_lens.to(DEV)

    def out(self):
        s = self.wl.spec
        n = self.q.shape[0]
        o = torch.full((n, s.hq, s.lv), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((n, s.hq), float("nan"), dtype=torch.float32, device=DEV)
        return o, lse

    def extend(self, cap=None, window=None, **mask_sinks):
        s = self.wl.spec
        o, lse = self.out()
        ws = pkx.extend_attention_fwd(
            self.q, self.k_extend, self.v_extend, o, self.k_buffer, self.v_buffer,
            self.qo_indptr, self.kv_indptr, self.kv_indices, self.wl.sm_scale,
            s.logit_cap if cap is None else cap,
            s.sliding_window if window is None else window, lse=lse, **_dev(mask_sinks))
        return o, lse, ws

    def ragged_paged(self, cap=None, window=None):
        s = self.wl.spec
        o, lse = self.out()
        ws = pkx.extend_attention_fwd_ragged_paged(
            self.q, self.k_extend, self.v_extend, o, self.k_buffer, self.v_buffer,
            self.qo_indptr, self.kv_indptr, self.kv_indices, self.wl.sm_scale,
            s.logit_cap if cap is None else cap,
            s.sliding_window if window is None else window, lse=lse)
        return o, lse, ws

    def unified(self, cap=None, window=None, scale=None, **mask_sinks):
        s = self.wl.spec
        uptr, uidx, plen = pkx.build_unified_kv_indices(
            self.kv_indptr, self.kv_indices, self.extend_start_loc, self.extend_seq_lens,
            self.extend_kv_indices, self.wl.batch)
        o, lse = self.out()
        ws = pkx.extend_attention_fwd_unified(
            self.q, o, self.k_buffer, self.v_buffer, self.qo_indptr, uptr, uidx, plen,
            self.wl.sm_scale if scale is None else scale, s.logit_cap if cap is None else cap,
            s.sliding_window if window is None else window, lse=lse, **_dev(mask_sinks))
        return o, lse, ws

    def decode(self, cap=None, window=None):
        s = self.wl.spec
        o, lse = self.out()
        ws = pkx.decode_attention_fwd(
            self.q, o, self.k_buffer, self.v_buffer, self.kv_indptr, self.kv_indices,
            self.wl.sm_scale, s.logit_cap if cap is None else cap,
            s.sliding_window if window is None else window, lse=lse)
        return o, lse, ws


def _dev(kw):
    """custom_mask / mask_indptr / sinks moved to the GPU (sinks as fp32)."""
    out = {}
    for k, v in kw.items():
        if v is None:
            continue
        v = v.to(DEV)
        out[k] = v.float() if k == "sinks" else v
    return out


def oracle_extend(wl: W.Workload, cap=None, window=None, rows=None, scale=None, **mask_sinks):
    s = wl.spec
    k_ext, v_ext = wl.extend_kv()
    kb, vb = wl.pool()
    return oracle.extend_attention(
        wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr, wl.kv_indices,
        wl.sm_scale if scale is None else scale,
        s.logit_cap if cap is None else cap, s.sliding_window if window is None else window,
        rows=rows, **{k: (v.double() if k == "sinks" else v) for k, v in mask_sinks.items()
                      if v is not None})


def oracle_decode(wl: W.Workload, cap=None, window=None):
    s = wl.spec
    kb, vb = wl.pool()
    return oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                   s.logit_cap if cap is None else cap,
                                   s.sliding_window if window is None else window)


def assert_close(o, lse, ref_o, ref_lse, what=""):
    """bf16 o within MAX_ABS / MEAN_ABS of the oracle, lse within LSE_ABS
    (finite entries; -inf must match exactly)."""
    o = o.detach().double().cpu()
    lse = lse.detach().double().cpu()
    assert torch.isfinite(o).all(), f"{what}: non-finite output"
    err = (o - ref_o).abs()
    assert err.max().item() <= MAX_ABS, f"{what}: max|err| {err.max().item():.3e}"
    assert err.mean().item() <= MEAN_ABS, f"{what}: mean|err| {err.mean().item():.3e}"
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin), f"{what}: lse finiteness differs"
    if fin.any():
        lerr = (lse[fin] - ref_lse[fin]).abs().max().item()
        assert lerr <= LSE_ABS, f"{what}: lse|err| {lerr:.3e}"
    return err.max().item(), err.mean().item()


def sample_rows(n_tokens, hq, count, seed):
    g = torch.Generator().manual_seed(seed)
    total = n_tokens * hq
    if total <= count:
        return torch.arange(total, dtype=torch.int64)
    return torch.randperm(total, generator=g)[:count].sort().values


def random_masks(wl: W.Workload, seed, density=0.5):
    """A custom mask for every sequence, flat uint8 with int32 offsets: row i
    of sequence b (T_b keys) at mask_indptr[b] + i * T_b; prefix keys are
    visible with probability 0.9, extend keys with ``density``, and every
    row sees its own key."""
    g = torch.Generator().manual_seed(seed)
    flat, indptr = [], [0]
    for b in range(wl.batch):
        E, P = wl.extend_lens[b], wl.prefix_lens[b]
        T = P + E
        m = torch.rand(E, T, generator=g)
        thr = torch.full((T,), density)
        thr[:P] = 0.9
        m = m < thr
        m[torch.arange(E), P + torch.arange(E)] = True
        flat.append(m.to(torch.uint8).reshape(-1))
        indptr.append(indptr[-1] + E * T)
    return torch.cat(flat), torch.tensor(indptr, dtype=torch.int32)
