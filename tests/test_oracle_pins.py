"""Pins of the float64 oracle against things other than itself.

Each test checks one oracle function against a library routine, a closed
form, an invariant the pages fix, or a hand-derived fixture, so that a
plausible slip in the oracle (a dropped term, an off-by-one in a mask, a wrong
sign, a transposed operand, a wrong head mapping) fails at least one of them.
``tests/test_oracle_mutants.py`` plants such slips and checks exactly that.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_extend_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-10


def _spec(**kw):
    return W.small_spec(**kw)


def _run_oracle(wl, cap=None, window=None, rows=None):
    k_ext, v_ext = wl.extend_kv()
    kb, vb = wl.pool()
    s = wl.spec
    return oracle.extend_attention(
        wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr, wl.kv_indices,
        wl.sm_scale, s.logit_cap if cap is None else cap,
        s.sliding_window if window is None else window, rows=rows)


def _dense_reference(wl, cap, window, masks=None, sinks=None):
    """Second formulation with library primitives: per sequence, the full
    [E, T] score matrix by matmul, tanh cap, a boolean mask from explicit
    position tables, softmax and matmul.  Returns (o, lse) float64.

    masks: per sequence a bool [E, T] that replaces the causal table (the
    window still applies).  sinks [Hq]: an extra key per row whose score is
    the head's sink and whose value vector is zero."""
    s = wl.spec
    g = s.hq // s.hkv
    outs, lses = [], []
    for b in range(wl.batch):
        t0 = int(wl.token_offsets[b])
        T = wl.prefix_lens[b] + wl.extend_lens[b]
        E = wl.extend_lens[b]
        if E == 0:
            continue
        k = wl.k_rows[t0:t0 + T].double().repeat_interleave(g, dim=1)  # [T,Hq,Lq]
        v = wl.v_rows[t0:t0 + T].double().repeat_interleave(g, dim=1)
        q0 = int(wl.qo_indptr[b])
        q = wl.q[q0:q0 + E].double()                                     # [E,Hq,Lq]
        sc = torch.einsum("ehd,thd->het", q, k) * wl.sm_scale
        if cap > 0:
            sc = cap * torch.tanh(sc / cap)
        qpos = torch.arange(E).view(E, 1) + wl.prefix_lens[b]
        kpos = torch.arange(T).view(1, T)
        vis = kpos <= qpos if masks is None else masks[b].bool()
        if window > 0:
            vis = vis & (qpos - kpos <= window)
        sc = sc.masked_fill(~vis.unsqueeze(0), float("-inf"))
        if sinks is not None:
            extra = torch.as_tensor(sinks, dtype=torch.float64).view(-1, 1, 1).expand(-1, E, 1)
            sc = torch.cat([sc, extra], dim=-1)                          # [Hq,E,T+1]
            v = torch.cat([v, torch.zeros(1, v.shape[1], v.shape[2], dtype=v.dtype)])
        lse = torch.logsumexp(sc, dim=-1)                                # [Hq,E]
        o = torch.einsum("het,thd->ehd", torch.softmax(sc, dim=-1), v)
        outs.append(o)
        lses.append(lse.transpose(0, 1))
    return torch.cat(outs), torch.cat(lses)


# ------------------------------------------------------------ prefix = 0 case
@pytest.mark.parametrize("lq,lv,hq,hkv", [(64, 64, 4, 2), (128, 128, 8, 2), (96, 80, 6, 3),
                                          (192, 128, 4, 1), (288, 256, 2, 1)])
def test_no_prefix_is_torch_causal_sdpa(lq, lv, hq, hkv):
    """With no cached prefix, extend attention is plain causal attention
    (flashinfer_backend.py, forward_extend: the ragged result alone when no
    sequence has a prefix).  Library pin: torch SDPA, is_causal, float64."""
    wl = W.draw(_spec(batch=3, hq=hq, hkv=hkv, lq=lq, lv=lv, prefix=[0, 0, 0],
                      extend=[1, 7, 33], seed=11))
    o, _ = _run_oracle(wl, cap=0.0, window=-1)
    g = hq // hkv
    for b in range(wl.batch):
        a, e = int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1])
        q = wl.q[a:e].double().transpose(0, 1)[None]
        k = wl.k_rows[a:e].double().repeat_interleave(g, 1).transpose(0, 1)[None]
        v = wl.v_rows[a:e].double().repeat_interleave(g, 1).transpose(0, 1)[None]
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=wl.sm_scale)
        torch.testing.assert_close(o[a:e], ref[0].transpose(0, 1), rtol=0, atol=TOL)


def test_no_prefix_window_is_sdpa_band_mask():
    """Sliding window with no prefix: query i sees keys i-W .. i
    (extend_attention.py, _fwd_kernel_unified, sliding-window mask).  Library
    pin: SDPA with a band mask built by tril/triu."""
    W_ = 5
    wl = W.draw(_spec(batch=1, hq=2, hkv=1, lq=64, lv=64, prefix=[0], extend=[23], seed=3))
    o, _ = _run_oracle(wl, cap=0.0, window=W_)
    E = wl.extend_lens[0]
    band = torch.ones(E, E, dtype=torch.bool).tril().triu(-W_)
    q = wl.q.double().transpose(0, 1)[None]
    k = wl.k_rows.double().repeat_interleave(2, 1).transpose(0, 1)[None]
    v = wl.v_rows.double().repeat_interleave(2, 1).transpose(0, 1)[None]
    ref = F.scaled_dot_product_attention(q, k, v, attn_mask=band, scale=wl.sm_scale)
    torch.testing.assert_close(o, ref[0].transpose(0, 1), rtol=0, atol=TOL)


# ------------------------------------------------------- dense brute force
@pytest.mark.parametrize("cap,window,seed", [(0.0, -1, 1), (30.0, -1, 2), (0.0, 9, 3),
                                             (2.5, 40, 4), (0.5, 1, 5)])
def test_matches_dense_library_formulation(cap, window, seed):
    """Brute force on small ragged batches with prefix, GQA, cap and window:
    the oracle's per-key loops equal a dense matmul/tanh/mask/softmax
    formulation built from torch library routines."""
    wl = W.draw(_spec(batch=4, hq=6, hkv=2, lq=64, lv=32, prefix=[0, 13, 70, 4],
                      extend=[9, 1, 20, 0], seed=seed, std=2.0))
    o, lse = _run_oracle(wl, cap=cap, window=window)
    ro, rl = _dense_reference(wl, cap, window)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


def test_mla_shape_matches_dense_formulation():
    """MLA layout (Lq=576 = 512 latent + 64 rope, Lv=512, V = first 512 dims
    of K, one KV head): the score is the full 576-dim dot product."""
    wl = W.draw(_spec(batch=2, hq=4, hkv=1, lq=576, lv=512, prefix=[6, 0],
                      extend=[3, 4], seed=21, std=0.5, v_aliases_k=True,
                      sm_scale=1 / math.sqrt(192)))
    o, lse = _run_oracle(wl)
    ro, rl = _dense_reference(wl, 0.0, -1)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


@pytest.mark.parametrize("lq,lv,seed", [(192, 128, 31), (288, 256, 32)])
def test_split_head_dims_match_dense_formulation(lq, lv, seed):
    """The other split head dims (extend_attention.py, the Lq = 192 = 128 +
    64 and Lq = 288 = 256 + 32 cases): the score is the full Lq-dim dot
    product and V has its own Lv dims; prefix, GQA and cap as elsewhere."""
    wl = W.draw(_spec(batch=3, hq=4, hkv=2, lq=lq, lv=lv, prefix=[0, 9, 17],
                      extend=[5, 3, 1], seed=seed, std=0.7))
    o, lse = _run_oracle(wl, cap=20.0, window=-1)
    ro, rl = _dense_reference(wl, 20.0, -1)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


# ------------------------------------------------------ split invariance
@pytest.mark.parametrize("cap,window", [(0.0, -1), (30.0, -1), (0.0, 6)])
def test_any_prefix_split_equals_full_causal(cap, window):
    """redundant_attention (extend_attention.py): laying prefix and extend
    out contiguously and running full causal attention gives the extend rows.
    So for one sequence of T tokens, every cut c (prefix c, extend T-c) must
    give rows c..T-1 of the cut-0 result."""
    T = 29
    base = W.draw(_spec(batch=1, hq=4, hkv=2, lq=64, lv=64, prefix=[0], extend=[T], seed=8))
    # Whole sequence as extend (cut 0): reference rows.
    full_o, full_lse = _run_oracle(base, cap=cap, window=window)
    kb, vb = base.pool()
    slots = base.slots
    for c in [1, 5, 17, 28]:
        q = base.q[c:]
        k_ext, v_ext = base.k_rows[c:], base.v_rows[c:]
        qo = torch.tensor([0, T - c], dtype=torch.int32)
        kvp = torch.tensor([0, c], dtype=torch.int32)
        o, lse = oracle.extend_attention(q, k_ext, v_ext, kb, vb, qo, kvp, slots[:c],
                                         base.sm_scale, cap, window)
        torch.testing.assert_close(o, full_o[c:], rtol=0, atol=TOL)
        torch.testing.assert_close(lse, full_lse[c:], rtol=0, atol=TOL)


# ------------------------------------------------------------ closed forms
def test_zero_query_gives_mean_of_visible_values():
    """q = 0 makes every visible score 0: o is the plain mean of the visible
    values and lse = log(#visible).  Checked with and without a window."""
    wl = W.draw(_spec(batch=2, hq=2, hkv=1, lq=64, lv=64, prefix=[10, 0], extend=[4, 6], seed=4))
    wl.q.zero_()
    for window in (-1, 3):
        o, lse = _run_oracle(wl, cap=0.0, window=window)
        r = 0
        for b in range(wl.batch):
            t0, P = int(wl.token_offsets[b]), wl.prefix_lens[b]
            for i in range(wl.extend_lens[b]):
                qpos = P + i
                lo = 0 if window <= 0 else max(0, qpos - window)
                vis = wl.v_rows[t0 + lo: t0 + qpos + 1, 0].double()
                for h in range(2):
                    torch.testing.assert_close(o[r, h], vis.mean(0), rtol=0, atol=TOL)
                    assert abs(lse[r, h].item() - math.log(vis.shape[0])) < TOL
                r += 1


def test_constant_values_give_that_constant():
    """Softmax weights sum to one: if every V row is the same vector c, o = c
    whatever the scores."""
    wl = W.draw(_spec(batch=2, hq=4, hkv=2, lq=64, lv=64, prefix=[7, 3], extend=[5, 2], seed=6))
    c = torch.randn(64, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    wl.v_rows[:] = c
    o, _ = _run_oracle(wl, cap=30.0, window=4)
    torch.testing.assert_close(o, c.double().expand_as(o), rtol=0, atol=1e-12)


def test_one_and_two_visible_keys_closed_forms():
    """A query that sees a single key returns that key's V row, with lse its
    own score; with W = 1 a query sees exactly itself and the key before it,
    and the output is the sigmoid blend of the two V rows."""
    # One key visible: decode over a single-token sequence.
    wl = W.draw(_spec(batch=1, hq=2, hkv=1, lq=64, lv=64, prefix=[0], extend=[1], seed=9))
    kb, vb = wl.pool()
    o, lse = oracle.decode_attention(wl.q, kb, vb, torch.tensor([0, 1], dtype=torch.int32),
                                     wl.slots, wl.sm_scale)
    for h in range(2):
        torch.testing.assert_close(o[0, h], wl.v_rows[0, 0].double(), rtol=0, atol=TOL)
        s = wl.sm_scale * (wl.q[0, h].double() @ wl.k_rows[0, 0].double())
        assert abs(lse[0, h].item() - s.item()) < TOL
    # W = 1: two keys visible (self and the one before).  Hand-worked:
    # weights sigma(s_prev - s_self), sigma(s_self - s_prev).
    wl = W.draw(_spec(batch=1, hq=1, hkv=1, lq=64, lv=64, prefix=[4], extend=[3], seed=10))
    o, lse = _run_oracle(wl, cap=0.0, window=1)
    for i in range(3):
        qpos = 4 + i
        qv = wl.q[i, 0].double()
        s_self = wl.sm_scale * (qv @ wl.k_rows[qpos, 0].double()).item()
        s_prev = wl.sm_scale * (qv @ wl.k_rows[qpos - 1, 0].double()).item()
        w_prev = 1.0 / (1.0 + math.exp(s_self - s_prev))
        ref = w_prev * wl.v_rows[qpos - 1, 0].double() + (1 - w_prev) * wl.v_rows[qpos, 0].double()
        torch.testing.assert_close(o[i, 0], ref, rtol=0, atol=TOL)
        m = max(s_self, s_prev)
        assert abs(lse[i, 0].item() - (m + math.log(math.exp(s_self - m) + math.exp(s_prev - m)))) < TOL


def test_large_window_and_large_cap_change_nothing():
    """W >= T keeps every causal key; cap -> infinity makes cap*tanh(s/cap)
    -> s.  Both must reproduce the plain result."""
    wl = W.draw(_spec(batch=2, hq=4, hkv=2, lq=64, lv=64, prefix=[12, 30], extend=[9, 4], seed=12))
    o0, l0 = _run_oracle(wl, cap=0.0, window=-1)
    o1, l1 = _run_oracle(wl, cap=0.0, window=1000)
    torch.testing.assert_close(o1, o0, rtol=0, atol=TOL)
    torch.testing.assert_close(l1, l0, rtol=0, atol=TOL)
    o2, l2 = _run_oracle(wl, cap=1e9, window=-1)
    torch.testing.assert_close(o2, o0, rtol=0, atol=1e-9)
    torch.testing.assert_close(l2, l0, rtol=0, atol=1e-9)


def test_tiny_cap_flattens_scores():
    """cap -> 0 squeezes every score into (-cap, cap): the weights become
    uniform, o -> mean of visible V, lse -> log(#visible)."""
    wl = W.draw(_spec(batch=1, hq=2, hkv=1, lq=64, lv=64, prefix=[6], extend=[5], seed=13, std=3.0))
    cap = 1e-9
    o, lse = _run_oracle(wl, cap=cap, window=-1)
    for i in range(5):
        vis = wl.v_rows[: 6 + i + 1, 0].double()
        for h in range(2):
            torch.testing.assert_close(o[i, h], vis.mean(0), rtol=0, atol=1e-8)
            assert abs(lse[i, h].item() - math.log(vis.shape[0])) < 1e-8


def test_cap_two_key_closed_form():
    """With two visible keys the output is a sigmoid blend of their values;
    with the cap, the blend weight uses cap*tanh(score/cap)."""
    wl = W.draw(_spec(batch=1, hq=1, hkv=1, lq=64, lv=64, prefix=[1], extend=[1], seed=14, std=2.0))
    cap = 1.5
    o, _ = _run_oracle(wl, cap=cap, window=-1)
    qv = wl.q[0, 0].double()
    s = [cap * math.tanh(wl.sm_scale * (qv @ wl.k_rows[j, 0].double()).item() / cap) for j in (0, 1)]
    w0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    ref = w0 * wl.v_rows[0, 0].double() + (1 - w0) * wl.v_rows[1, 0].double()
    torch.testing.assert_close(o[0, 0], ref, rtol=0, atol=TOL)


def test_gqa_head_mapping():
    """q head h reads kv head h // (Hq/Hkv) (kv_group_num): zeroing every V
    row of kv head 1 must zero exactly q heads 2 and 3 when Hq=4, Hkv=2."""
    wl = W.draw(_spec(batch=1, hq=4, hkv=2, lq=64, lv=64, prefix=[5], extend=[4], seed=15))
    wl.v_rows[:, 1] = 0
    o, _ = _run_oracle(wl)
    assert torch.all(o[:, 2:] == 0)
    assert torch.all(o[:, :2].abs().sum(-1) > 0)


def test_sample_rows_equal_full_rows():
    """Row-sampled mode returns exactly the rows of the full run."""
    wl = W.draw(_spec(batch=3, hq=4, hkv=2, lq=64, lv=64, prefix=[3, 0, 9], extend=[2, 5, 3], seed=16))
    o, lse = _run_oracle(wl, cap=5.0, window=4)
    rows = [0, 5, 17, 39, 22]
    so, sl = _run_oracle(wl, cap=5.0, window=4, rows=rows)
    hq = 4
    for r, row in enumerate(rows):
        assert torch.equal(so[r], o[row // hq, row % hq])
        assert sl[r] == lse[row // hq, row % hq]


# --------------------------------------------------------------------- decode
def test_decode_equals_extend_of_last_token():
    """Decode (flashinfer_backend.py, forward_decode: the token's K/V are
    saved first, then one query attends to all T keys) equals extend with
    prefix T-1 and the last token as the one extend token."""
    wl = W.draw(W.WorkloadSpec("dec", batch=3, hq=8, hkv=2, lq=128, lv=128,
                               prefix=[0, 6, 40], extend=[1, 1, 1], num_slots=128,
                               seed=17, decode=True))
    kb, vb = wl.pool()
    o, lse = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     logit_cap=4.0, sliding_window=5)
    for b in range(3):
        T = wl.prefix_lens[b] + 1
        t0 = int(wl.token_offsets[b])
        slots = wl.slots[t0:t0 + T]
        eo, el = oracle.extend_attention(
            wl.q[b:b + 1], wl.k_rows[t0 + T - 1:t0 + T], wl.v_rows[t0 + T - 1:t0 + T], kb, vb,
            torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0, T - 1], dtype=torch.int32),
            slots[:T - 1], wl.sm_scale, 4.0, 5)
        torch.testing.assert_close(o[b], eo[0], rtol=0, atol=TOL)
        torch.testing.assert_close(lse[b], el[0], rtol=0, atol=TOL)


def test_decode_window_keeps_last_w_plus_one_keys():
    """Sliding-window decode keeps min(T, W+1) keys (flashinfer_backend.py,
    sliding-window decode index updater): equal to plain decode over only
    the last W+1 slots."""
    wl = W.draw(W.WorkloadSpec("dec", batch=2, hq=4, hkv=1, lq=64, lv=64,
                               prefix=[20, 3], extend=[1, 1], num_slots=64, seed=18, decode=True))
    kb, vb = wl.pool()
    Wn = 6
    o, lse = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     sliding_window=Wn)
    sub_idx, sub_ptr = [], [0]
    for b in range(2):
        a, e = int(wl.kv_indptr[b]), int(wl.kv_indptr[b + 1])
        keep = wl.kv_indices[max(a, e - (Wn + 1)):e]
        sub_idx.append(keep)
        sub_ptr.append(sub_ptr[-1] + keep.numel())
    o2, l2 = oracle.decode_attention(wl.q, kb, vb, torch.tensor(sub_ptr, dtype=torch.int32),
                                     torch.cat(sub_idx), wl.sm_scale)
    torch.testing.assert_close(o, o2, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, l2, rtol=0, atol=TOL)


def test_empty_sequences_are_harmless():
    """Padding sequences (length 0, as the CUDA-graph runner pads with
    seq_len 0) produce no rows and do not disturb their neighbours."""
    a = W.draw(_spec(batch=3, hq=4, hkv=2, lq=64, lv=64, prefix=[4, 0, 6], extend=[3, 0, 2], seed=19))
    o, lse = _run_oracle(a)
    assert o.shape[0] == 5
    ro, rl = _dense_reference(a, 0.0, -1)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    kb, vb = a.pool()
    od, ld = oracle.decode_attention(a.q[:2], kb, vb, torch.tensor([0, 0, 0], dtype=torch.int32),
                                     torch.zeros(0, dtype=torch.int32), a.sm_scale)
    assert torch.all(od == 0) and torch.all(torch.isneginf(ld))


# ---------------------------------------------------------------- merge_state
def test_merge_of_two_key_halves_equals_attention_over_all():
    """merge_state of attention over key set A and over key set B equals
    attention over A u B (flashinfer_backend.py, forward_extend: ragged
    extend result merged with the non-causal paged prefix result).  The
    partial outputs are rounded to bf16 before merging, so the bound is the
    largest rounding error of the merged inputs (a convex combination cannot
    amplify it) plus fp32 rounding of the lse inputs."""
    wl = W.draw(W.WorkloadSpec("dec", batch=4, hq=8, hkv=2, lq=128, lv=128,
                               prefix=[9, 30, 1, 63], extend=[1, 1, 1, 1], num_slots=256,
                               seed=20, decode=True))
    kb, vb = wl.pool()
    full_o, full_l = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale)
    ia, ib, pa, pb = [], [], [0], [0]
    for b in range(4):
        a, e = int(wl.kv_indptr[b]), int(wl.kv_indptr[b + 1])
        cut = a + (e - a) // 3
        ia.append(wl.kv_indices[a:cut]); ib.append(wl.kv_indices[cut:e])
        pa.append(pa[-1] + cut - a); pb.append(pb[-1] + e - cut)
    oa, la = oracle.decode_attention(wl.q, kb, vb, torch.tensor(pa, dtype=torch.int32),
                                     torch.cat(ia), wl.sm_scale)
    ob, lb = oracle.decode_attention(wl.q, kb, vb, torch.tensor(pb, dtype=torch.int32),
                                     torch.cat(ib), wl.sm_scale)
    va, vb_ = oa.to(torch.bfloat16), ob.to(torch.bfloat16)
    v, s = oracle.merge_state(va, la.float(), vb_, lb.float())
    bound = max((va.double() - oa).abs().max().item(), (vb_.double() - ob).abs().max().item())
    assert (v - full_o).abs().max().item() <= bound + 1e-6
    torch.testing.assert_close(s, full_l, rtol=0, atol=1e-5)


def test_merge_closed_forms():
    """An empty side (lse = -inf) has weight 0; equal lse halves average
    and add log 2; both empty gives 0 and -inf."""
    g = torch.Generator().manual_seed(2)
    va = torch.randn(3, 2, 16, generator=g).to(torch.bfloat16)
    vb = torch.randn(3, 2, 16, generator=g).to(torch.bfloat16)
    sa = torch.tensor([[float("-inf"), 1.0], [0.5, float("-inf")], [float("-inf"), -2.0]])
    sb = torch.tensor([[0.25, 1.0], [float("-inf"), float("-inf")], [3.0, -2.0]])
    v, s = oracle.merge_state(va, sa, vb, sb)
    torch.testing.assert_close(v[0, 0], vb[0, 0].double(), rtol=0, atol=0)
    assert s[0, 0] == 0.25
    torch.testing.assert_close(v[0, 1], (va[0, 1].double() + vb[0, 1].double()) / 2, rtol=0, atol=1e-15)
    assert abs(s[0, 1].item() - (1.0 + math.log(2))) < 1e-15
    torch.testing.assert_close(v[1, 0], va[1, 0].double(), rtol=0, atol=0)
    assert torch.all(v[1, 1] == 0) and torch.isneginf(s[1, 1])
    torch.testing.assert_close(v[2, 0], vb[2, 0].double(), rtol=0, atol=0)


def test_merge_weights_are_softmax_of_lse():
    """Library pin: the merged value equals softmax([s_a, s_b]) . [v_a, v_b]
    and the merged lse equals torch.logsumexp([s_a, s_b])."""
    g = torch.Generator().manual_seed(3)
    va = torch.randn(50, 4, 32, generator=g).to(torch.bfloat16)
    vb = torch.randn(50, 4, 32, generator=g).to(torch.bfloat16)
    sa = torch.randn(50, 4, generator=g) * 10
    sb = torch.randn(50, 4, generator=g) * 10
    v, s = oracle.merge_state(va, sa, vb, sb)
    st = torch.stack([sa.double(), sb.double()], -1)
    w = torch.softmax(st, -1)
    ref = w[..., :1] * va.double() + w[..., 1:] * vb.double()
    torch.testing.assert_close(v, ref, rtol=0, atol=1e-12)
    torch.testing.assert_close(s, torch.logsumexp(st, -1), rtol=0, atol=1e-12)


# ------------------------------------------------------------ unified indices
def test_unified_indices_hand_fixture():
    """Hand-derived worked example (tests/golden/unified_indices_hand.json)."""
    with open(os.path.join(GOLDEN, "unified_indices_hand.json")) as f:
        fx = json.load(f)
    i, e = fx["inputs"], fx["expected"]
    t = lambda k: torch.tensor(i[k], dtype=torch.int32)
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        t("prefix_kv_indptr"), t("prefix_kv_indices"), t("extend_start_loc"),
        t("extend_seq_lens"), t("extend_kv_indices"), i["bs"], fill=-7)
    assert uptr.tolist() == e["unified_kv_indptr"]
    n = e["unified_kv_indptr"][-1]
    assert uidx[:n].tolist() == e["unified_kv_indices_prefix"]
    assert torch.all(uidx[n:] == -7)
    assert plen.tolist() == e["prefix_lens"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_unified_indices_are_per_sequence_concatenation(seed):
    """Random ragged batches with arbitrary extend_start_loc: the unified
    list equals numpy concatenation of each sequence's prefix slice and
    extend slice, the indptr equals numpy cumsum, bit for bit."""
    rng = np.random.default_rng(seed)
    bs = int(rng.integers(1, 40))
    plens = rng.integers(0, 300, bs)
    plens[rng.random(bs) < 0.2] = 0
    elens = rng.integers(0, 200, bs)
    pptr = np.concatenate([[0], np.cumsum(plens)]).astype(np.int32)
    pidx = rng.integers(0, 2**31 - 1, int(plens.sum())).astype(np.int32)
    # extend buffer in a shuffled order with gaps
    order = rng.permutation(bs)
    starts = np.zeros(bs, np.int64)
    pos = 0
    for b in order:
        pos += int(rng.integers(0, 4))
        starts[b] = pos
        pos += int(elens[b])
    eidx = rng.integers(0, 2**31 - 1, pos + 3).astype(np.int32)
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        torch.from_numpy(pptr), torch.from_numpy(pidx), torch.from_numpy(starts.astype(np.int32)),
        torch.from_numpy(elens.astype(np.int32)), torch.from_numpy(eidx), bs, fill=-1)
    ref = np.concatenate([np.concatenate([pidx[pptr[b]:pptr[b + 1]],
                                          eidx[starts[b]:starts[b] + elens[b]]])
                          for b in range(bs)]).astype(np.int64)
    n = int(plens.sum() + elens.sum())
    assert np.array_equal(uidx[:n].numpy(), ref)
    assert torch.all(uidx[n:] == -1)
    assert np.array_equal(uptr.numpy(), np.concatenate([[0], np.cumsum(plens + elens)]))
    assert np.array_equal(plen.numpy(), plens)


def test_two_stage_equals_unified():
    """The two-stage form (prefix through indices, extend contiguous) and the
    unified form (everything through unified indices) compute the same
    thing on the same data (extend_attention.py: extend_attention_fwd vs
    extend_attention_fwd_unified)."""
    wl = W.draw(_spec(batch=4, hq=8, hkv=2, lq=128, lv=128, prefix=[0, 17, 3, 60],
                      extend=[12, 1, 0, 33], seed=22))
    o, lse = _run_oracle(wl, cap=20.0, window=15)
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    kb, vb = wl.pool()
    uo, ul = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, 20.0, 15)
    assert torch.equal(o, uo) and torch.equal(lse, ul)


def test_default_scale_is_inverse_sqrt_lq():
    """sm_scale <= 0 means 1/sqrt(Lq) (the launcher's 'sm_scale or
    1/sqrt(Lq)')."""
    wl = W.draw(_spec(batch=1, hq=2, hkv=1, lq=64, lv=64, prefix=[3], extend=[2], seed=23))
    k_ext, v_ext = wl.extend_kv()
    kb, vb = wl.pool()
    args = (wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr, wl.kv_indices)
    o0, _ = oracle.extend_attention(*args, 0.0)
    o1, _ = oracle.extend_attention(*args, 1.0 / 8.0)
    assert torch.equal(o0, o1)


# --------------------------------------------- custom mask and attention sinks
def _random_masks(wl, seed, density=0.4):
    """Per sequence a random bool [E, T] (each row also sees its own key),
    and the flat uint8 layout with per-sequence offsets: row i of sequence b
    at mask_indptr[b] + i * T_b."""
    g = torch.Generator().manual_seed(seed)
    masks, flat, indptr = [], [], [0]
    for b in range(wl.batch):
        E, P = wl.extend_lens[b], wl.prefix_lens[b]
        T = P + E
        m = torch.rand(E, T, generator=g) < density
        m[torch.arange(E), P + torch.arange(E)] = True
        masks.append(m)
        flat.append(m.to(torch.uint8).reshape(-1))
        indptr.append(indptr[-1] + E * T)
    return masks, torch.cat(flat), torch.tensor(indptr, dtype=torch.int32)


def _run_masked(wl, masks_flat=None, mask_indptr=None, sinks=None, cap=None, window=None):
    k_ext, v_ext = wl.extend_kv()
    kb, vb = wl.pool()
    s = wl.spec
    return oracle.extend_attention(
        wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr, wl.kv_indices,
        wl.sm_scale, s.logit_cap if cap is None else cap,
        s.sliding_window if window is None else window,
        custom_mask=masks_flat, mask_indptr=mask_indptr, sinks=sinks)


@pytest.mark.parametrize("cap,window,seed", [(0.0, -1, 1), (15.0, -1, 2), (0.0, 9, 3)])
def test_custom_mask_matches_dense_formulation(cap, window, seed):
    """A custom mask replaces the causal mask and keeps the window (sglang
    extend_attention.py, _fwd_kernel_unified: "Apply custom mask", causal
    only when not USE_CUSTOM_MASK): brute-force dense formulation."""
    wl = W.draw(_spec(batch=3, hq=6, hkv=2, lq=64, lv=32, prefix=[0, 21, 7],
                      extend=[11, 6, 30], seed=seed, std=2.0))
    masks, flat, indptr = _random_masks(wl, seed)
    o, lse = _run_masked(wl, flat, indptr, cap=cap, window=window)
    ro, rl = _dense_reference(wl, cap, window, masks=masks)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


def test_causal_pattern_mask_equals_no_mask():
    """A mask that spells out the causal pattern gives the unmasked result."""
    wl = W.draw(_spec(batch=2, hq=4, hkv=2, lq=64, lv=64, prefix=[5, 40], extend=[9, 17], seed=4))
    flat, indptr = [], [0]
    for b in range(wl.batch):
        E, P = wl.extend_lens[b], wl.prefix_lens[b]
        m = torch.arange(P + E).view(1, -1) <= (P + torch.arange(E)).view(-1, 1)
        flat.append(m.to(torch.uint8).reshape(-1))
        indptr.append(indptr[-1] + E * (P + E))
    o, lse = _run_masked(wl, torch.cat(flat), torch.tensor(indptr, dtype=torch.int32))
    ro, rl = _run_oracle(wl)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


def test_all_ones_mask_is_non_causal_sdpa():
    """An all-ones mask on a sequence without prefix is plain non-causal
    attention: torch's scaled_dot_product_attention(is_causal=False)."""
    wl = W.draw(_spec(batch=1, hq=4, hkv=2, lq=64, lv=64, prefix=[0], extend=[23], seed=12))
    E = wl.extend_lens[0]
    flat = torch.ones(E * E, dtype=torch.uint8)
    o, _ = _run_masked(wl, flat, torch.tensor([0, E * E], dtype=torch.int32))
    q = wl.q.double().transpose(0, 1)                                   # [Hq,E,D]
    k = wl.k_rows[:E].double().repeat_interleave(2, dim=1).transpose(0, 1)
    v = wl.v_rows[:E].double().repeat_interleave(2, dim=1).transpose(0, 1)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=False, scale=wl.sm_scale)
    torch.testing.assert_close(o, ref.transpose(0, 1), rtol=0, atol=TOL)


@pytest.mark.parametrize("window", [-1, 7])
def test_sinks_match_an_extra_zero_valued_key(window):
    """A sink logit per head adds exp(sink - m) to the denominator only
    (sglang extend_attention.py, "Handle sink tokens"): the same as one more
    key per row whose score is the sink and whose value vector is zero."""
    wl = W.draw(_spec(batch=3, hq=6, hkv=3, lq=64, lv=32, prefix=[0, 12, 50],
                      extend=[8, 15, 4], seed=17, std=1.5))
    sinks = torch.tensor([-1.0, 0.5, 2.0, 4.0, -3.0, 1.25], dtype=torch.float64)
    o, lse = _run_masked(wl, sinks=sinks, window=window)
    ro, rl = _dense_reference(wl, 0.0, window, sinks=sinks)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


def test_sink_with_one_visible_key_closed_form():
    """Window 0 leaves each row its own key only: o = v_self * e^s / (e^s +
    e^sink), lse = log(e^s + e^sink)."""
    wl = W.draw(_spec(batch=1, hq=2, hkv=1, lq=64, lv=64, prefix=[3], extend=[5], seed=6))
    sinks = torch.tensor([0.7, -0.4], dtype=torch.float64)
    # window 0 is "off"; a window of 1e-9 is not an integer: use the mask
    E, P = 5, 3
    m = torch.zeros(E, P + E, dtype=torch.bool)
    m[torch.arange(E), P + torch.arange(E)] = True
    o, lse = _run_masked(wl, m.to(torch.uint8).reshape(-1),
                         torch.tensor([0, E * (P + E)], dtype=torch.int32), sinks=sinks)
    for i in range(E):
        for h in range(2):
            k = wl.k_rows[P + i, 0].double()
            v = wl.v_rows[P + i, 0].double()
            sc = float(wl.sm_scale * (wl.q[i, h].double() * k).sum())
            w = math.exp(sc) / (math.exp(sc) + math.exp(float(sinks[h])))
            torch.testing.assert_close(o[i, h], v * w, rtol=0, atol=1e-12)
            assert abs(float(lse[i, h]) - math.log(math.exp(sc) + math.exp(float(sinks[h])))) < 1e-12


def test_very_negative_sinks_change_nothing():
    wl = W.draw(_spec(batch=2, hq=4, hkv=2, lq=64, lv=64, prefix=[10, 0], extend=[6, 9], seed=9))
    o, lse = _run_masked(wl, sinks=torch.full((4,), -1e4, dtype=torch.float64))
    ro, rl = _run_oracle(wl)
    torch.testing.assert_close(o, ro, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, rl, rtol=0, atol=TOL)


# ------------------------------- KV-index gather and KV write into the pool
def _gather(table, rpi, lens, start=None):
    t = lambda x: torch.tensor(x, dtype=torch.int64) if x is not None else None
    return oracle.create_kv_indices(torch.tensor(table, dtype=torch.int32),
                                    t(rpi), t(lens), t(start))


def test_kv_indices_hand_fixture():
    """Hand-derived worked example (tests/golden/kv_indices_hand.json),
    with and without kv_start_idx."""
    with open(os.path.join(GOLDEN, "kv_indices_hand.json")) as f:
        fx = json.load(f)
    for name, c in fx["cases"].items():
        kvp, kvi = _gather(fx["req_to_token"], c["req_pool_indices"],
                           c["paged_kernel_lens"], c["kv_start_idx"])
        assert kvp.tolist() == c["expected_kv_indptr"], name
        assert kvi.tolist() == c["expected_kv_indices"], name


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_kv_indices_are_row_slices(seed):
    """Random tables, rows and windows: kv_indices equals numpy
    concatenation of the row slices [kv_start, kv_start + len), kv_indptr
    equals numpy's running sum, bit for bit."""
    rng = np.random.default_rng(seed)
    rows, cols, bs = 9, 300, 6
    table = rng.integers(0, 1 << 30, size=(rows, cols), dtype=np.int32)
    rpi = rng.choice(rows, size=bs, replace=False)
    lens = rng.integers(0, 120, size=bs)
    lens[seed % bs] = 0
    start = rng.integers(0, cols - 120, size=bs)
    for st in (None, start):
        kvp, kvi = oracle.create_kv_indices(torch.from_numpy(table), torch.from_numpy(rpi),
                                            torch.from_numpy(lens),
                                            torch.from_numpy(st) if st is not None else None)
        s0 = st if st is not None else np.zeros(bs, dtype=np.int64)
        want = np.concatenate([table[rpi[b], s0[b]:s0[b] + lens[b]] for b in range(bs)])
        assert np.array_equal(kvi.numpy(), want)
        assert np.array_equal(kvp.numpy(), np.concatenate([[0], np.cumsum(lens)]))


def test_whole_sequence_gather_is_the_unified_index_list():
    """With paged_kernel_lens = seq_lens and no start (the full-attention
    prefill updater), the gather from a table holding each sequence's
    prefix then extend slots is the unified index list of
    build_unified_kv_indices."""
    wl = W.draw(_spec(batch=4, hq=4, hkv=2, lq=64, lv=64, prefix=[9, 0, 31, 2],
                      extend=[4, 7, 0, 1], seed=41))
    table, rpi, seq = wl.req_to_token(seed=3)
    kvp, kvi = oracle.create_kv_indices(table, rpi, seq)
    uptr, uidx, _ = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    assert torch.equal(kvp, uptr)
    assert torch.equal(kvi.to(torch.int64), uidx)


@pytest.mark.parametrize("window", [1, 5, 40])
def test_window_start_keeps_the_extend_window(window):
    """The sliding-window prefill updater gathers only the last
    min(T, W + E) slots (kv_start = T - that); extend attention with window W
    over those keys equals extend attention with window W over all keys."""
    wl = W.draw(_spec(batch=3, hq=4, hkv=2, lq=64, lv=64, prefix=[30, 0, 12],
                      extend=[6, 9, 3], seed=42))
    table, rpi, seq = wl.req_to_token(seed=4)
    ext = torch.tensor(wl.extend_lens, dtype=torch.int64)
    pre = seq - ext
    paged = torch.minimum(seq, window + seq - pre)
    kvp, kvi = oracle.create_kv_indices(table, rpi, paged, seq - paged)
    kb, vb = wl.pool()
    o, lse = oracle.extend_attention_unified(
        wl.q, kb, vb, wl.qo_indptr, kvp, kvi, (paged - ext).to(torch.int32),
        wl.sm_scale, 0.0, window)
    fp, fi = oracle.create_kv_indices(table, rpi, seq)
    o2, l2 = oracle.extend_attention_unified(
        wl.q, kb, vb, wl.qo_indptr, fp, fi, pre.to(torch.int32), wl.sm_scale, 0.0, window)
    torch.testing.assert_close(o, o2, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, l2, rtol=0, atol=TOL)


def test_window_start_keeps_the_decode_window():
    """The sliding-window decode updater gathers the last min(T, W + 1)
    slots; plain decode over them equals windowed decode over all slots."""
    wl = W.draw(W.WorkloadSpec("dec", batch=3, hq=4, hkv=2, lq=64, lv=64,
                               prefix=[25, 2, 0], extend=[1, 1, 1], num_slots=96, seed=43,
                               decode=True))
    table, rpi, seq = wl.req_to_token(seed=5)
    kb, vb = wl.pool()
    Wn = 7
    paged = torch.clamp(seq, max=Wn + 1)
    kvp, kvi = oracle.create_kv_indices(table, rpi, paged, seq - paged)
    o, lse = oracle.decode_attention(wl.q, kb, vb, kvp, kvi, wl.sm_scale)
    fp, fi = oracle.create_kv_indices(table, rpi, seq)
    o2, l2 = oracle.decode_attention(wl.q, kb, vb, fp, fi, wl.sm_scale, sliding_window=Wn)
    torch.testing.assert_close(o, o2, rtol=0, atol=TOL)
    torch.testing.assert_close(lse, l2, rtol=0, atol=TOL)


def test_set_kv_buffer_hand_fixture():
    """Hand-derived worked example (tests/golden/set_kv_buffer_hand.json)."""
    with open(os.path.join(GOLDEN, "set_kv_buffer_hand.json")) as f:
        fx = json.load(f)
    bf = lambda x: torch.tensor(x, dtype=torch.bfloat16)
    kb = torch.full((fx["num_slots"], 2, 2), fx["fill"], dtype=torch.bfloat16)
    vb = kb.clone()
    k2, v2 = oracle.set_kv_buffer(kb, vb, torch.tensor(fx["cache_loc"]), bf(fx["k"]), bf(fx["v"]))
    assert torch.equal(k2, bf(fx["expected_k_buffer"]))
    assert torch.equal(v2, bf(fx["expected_v_buffer"]))


@pytest.mark.parametrize("hkv,lk,lv,k_only", [(2, 64, 64, False), (3, 128, 96, False),
                                              (1, 576, 512, True)])
def test_set_kv_buffer_matches_index_copy(hkv, lk, lv, k_only):
    """Random pools, distinct random slots and strided inputs (every head
    row taken from a wider tensor): the write equals torch index_copy_ of the
    token rows into the pool, and no other slot changes."""
    g = torch.Generator().manual_seed(44 + lk)
    slots, n = 50, 17
    kb = torch.randn(slots, hkv, lk, generator=g).to(torch.bfloat16)
    vb = torch.randn(slots, hkv, lv, generator=g).to(torch.bfloat16)
    loc = torch.randperm(slots, generator=g)[:n]
    k = torch.randn(n, hkv + 1, lk + 8, generator=g).to(torch.bfloat16)[:, 1:, 8:]
    v = torch.randn(n, hkv, 2 * lv, generator=g).to(torch.bfloat16)[:, :, :lv]
    k2, v2 = oracle.set_kv_buffer(kb, vb, loc, k, None if k_only else v)
    assert torch.equal(k2, kb.clone().index_copy_(0, loc, k.contiguous()))
    assert torch.equal(v2, vb if k_only else vb.clone().index_copy_(0, loc, v.contiguous()))


def test_written_pool_gives_the_two_stage_result():
    """Extend slots holding stale data, then set_kv_buffer of k_extend and
    v_extend at out_cache_loc (the extend slots): unified attention over the
    written pool equals the two-stage form, which reads the extend K/V
    directly (forward_extend writes the pool before the paged pass)."""
    wl = W.draw(_spec(batch=3, hq=8, hkv=2, lq=128, lv=128, prefix=[11, 0, 40],
                      extend=[5, 13, 2], seed=45))
    o, lse = _run_oracle(wl)
    kb, vb = wl.pool()
    loc = wl.extend_kv_indices.to(torch.int64)
    g = torch.Generator().manual_seed(9)
    kb[loc] = torch.randn(kb[loc].shape, generator=g).to(torch.bfloat16)
    vb[loc] = torch.randn(vb[loc].shape, generator=g).to(torch.bfloat16)
    k_ext, v_ext = wl.extend_kv()
    kb2, vb2 = oracle.set_kv_buffer(kb, vb, loc, k_ext, v_ext)
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    uo, ul = oracle.extend_attention_unified(wl.q, kb2, vb2, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, 0.0, -1)
    assert torch.equal(o, uo) and torch.equal(lse, ul)


# ------------------------------------------------------------- fp8 KV pool
FP8 = [(oracle.KV_E4M3, torch.float8_e4m3fn, 448.0), (oracle.KV_E5M2, torch.float8_e5m2, 57344.0)]


@pytest.mark.parametrize("fmt,dt,_max", FP8)
def test_fp8_code_values_match_torch(fmt, dt, _max):
    """Every one of the 256 codes decodes to torch's own float8 value (NaN
    where torch has NaN, +-inf for e5m2's infinities)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = codes.view(dt).to(torch.float64)
    got = torch.tensor([oracle.fp8_value(c, fmt) for c in range(256)], dtype=torch.float64)
    assert torch.equal(torch.isnan(got), torch.isnan(want))
    ok = ~torch.isnan(want)
    assert torch.equal(got[ok], want[ok])


@pytest.mark.parametrize("fmt,dt,vmax", FP8)
def test_fp8_rounding_matches_torch_in_range(fmt, dt, vmax):
    """In range, the code of an fp32 value is torch's round-to-nearest-even
    conversion: random values over many binades, every midpoint between two
    neighbouring codes (the ties), the subnormal range and signed zeros."""
    g = torch.Generator().manual_seed(61)
    vals = [torch.randn(4000, generator=g) * s for s in (1e-4, 1e-2, 0.3, 3.0, 60.0)]
    finite = [oracle.fp8_value(c, fmt) for c in range(128)]
    finite = sorted(v for v in finite if math.isfinite(v))
    mids = [(a + b) / 2 for a, b in zip(finite, finite[1:])]
    vals.append(torch.tensor(mids + [-m for m in mids] + [0.0, -0.0, vmax, -vmax]))
    x = torch.cat(vals).to(torch.float32)
    x = x[x.abs() <= vmax]
    want = x.to(dt).view(torch.uint8).to(torch.int64)
    got = torch.tensor([oracle.fp8_code(float(v), fmt) for v in x], dtype=torch.int64)
    assert torch.equal(got, want)


@pytest.mark.parametrize("fmt,dt,vmax", FP8)
def test_fp8_saturates_past_the_largest_code(fmt, dt, vmax):
    top = [c for c in range(128) if oracle.fp8_value(c, fmt) == vmax][0]
    for x in (vmax * 1.01, vmax * 4, 1e30, float("inf")):
        assert oracle.fp8_code(x, fmt) == top
        assert oracle.fp8_code(-x, fmt) == top | 0x80


def _fp8_pool_pair(wl, fmt, k_scale, v_scale):
    """The workload's pool quantized into fp8 through the oracle's KV write,
    and the same pool dequantized into bf16 (exact: a code times a power of
    two fits in bf16)."""
    kb, vb = wl.pool()
    dt = dict((f, d) for f, d, _ in FP8)[fmt]
    z8k = torch.zeros(kb.shape, dtype=torch.uint8).view(dt)
    z8v = torch.zeros(vb.shape, dtype=torch.uint8).view(dt)
    loc = wl.slots.to(torch.int64)
    k8, v8 = oracle.set_kv_buffer_fp8(z8k, z8v, loc, wl.k_rows, wl.v_rows, k_scale, v_scale)
    kdq = (k8.to(torch.float64) * k_scale).to(torch.bfloat16)
    vdq = (v8.to(torch.float64) * v_scale).to(torch.bfloat16)
    assert torch.equal(kdq.double(), k8.to(torch.float64) * k_scale)  # exact
    return k8, v8, kdq, vdq


@pytest.mark.parametrize("fmt", [oracle.KV_E4M3, oracle.KV_E5M2])
def test_fp8_pool_attention_equals_bf16_pool_of_its_values(fmt):
    """With power-of-two scales every dequantized element is a bf16 value;
    two-stage, unified and decode attention over the fp8 pool (k_scale,
    v_scale) equal the same attention over that bf16 pool, bit for bit."""
    ks, vs = 0.25, 4.0
    wl = W.draw(_spec(batch=3, hq=8, hkv=2, lq=64, lv=64, prefix=[20, 0, 45],
                      extend=[6, 9, 3], seed=62))
    k8, v8, kdq, vdq = _fp8_pool_pair(wl, fmt, ks, vs)
    k_ext, v_ext = wl.extend_kv()
    s = wl.spec
    args = (wl.qo_indptr, wl.kv_indptr, wl.kv_indices, wl.sm_scale, 10.0, 30)
    o8, l8 = oracle.extend_attention(wl.q, k_ext, v_ext, k8, v8, *args, k_scale=ks, v_scale=vs)
    ob, lb = oracle.extend_attention(wl.q, k_ext, v_ext, kdq, vdq, *args)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    o8, l8 = oracle.extend_attention_unified(wl.q, k8, v8, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, 0.0, -1, k_scale=ks, v_scale=vs)
    ob, lb = oracle.extend_attention_unified(wl.q, kdq, vdq, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, 0.0, -1)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)
    q1 = wl.q[:3]
    o8, l8 = oracle.decode_attention(q1, k8, v8, uptr, uidx.to(torch.int32), wl.sm_scale,
                                     k_scale=ks, v_scale=vs)
    ob, lb = oracle.decode_attention(q1, kdq, vdq, uptr, uidx.to(torch.int32), wl.sm_scale)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)


def test_fp8_write_matches_torch_quantization():
    """The fp8 KV write equals torch: (k.float() / scale).to(float8) at the
    slots (values kept in range), other slots unchanged."""
    g = torch.Generator().manual_seed(63)
    n, hkv, d, slots = 13, 2, 64, 40
    k = (torch.randn(n, hkv, d, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(n, hkv, d, generator=g) * 3).to(torch.bfloat16)
    loc = torch.randperm(slots, generator=g)[:n]
    for fmt, dt, _ in FP8:
        kb = torch.randint(0, 120, (slots, hkv, d), generator=g, dtype=torch.uint8).view(dt)
        vb = torch.randint(0, 120, (slots, hkv, d), generator=g, dtype=torch.uint8).view(dt)
        k2, v2 = oracle.set_kv_buffer_fp8(kb, vb, loc, k, v, 0.5, 2.0)
        wk = kb.view(torch.uint8).clone()
        wk[loc] = (k.float() / 0.5).to(dt).view(torch.uint8)
        wv = vb.view(torch.uint8).clone()
        wv[loc] = (v.float() / 2.0).to(dt).view(torch.uint8)
        assert torch.equal(k2.view(torch.uint8), wk)
        assert torch.equal(v2.view(torch.uint8), wv)


# ------------------------------------------------------ paged KV (page size > 1)
def test_paged_indices_hand_fixture():
    """Hand-derived worked example (tests/golden/paged_indices_hand.json)."""
    with open(os.path.join(GOLDEN, "paged_indices_hand.json")) as f:
        fx = json.load(f)
    t = lambda k: torch.tensor(fx[k], dtype=torch.int32)
    tptr, tidx = oracle.expand_paged_kv_indices(t("kv_indptr"), t("kv_indices"),
                                                t("kv_last_page_len"), fx["page_size"])
    assert tptr.tolist() == fx["expected_token_indptr"]
    assert tidx.tolist() == fx["expected_token_indices"]


def test_page_size_one_is_the_identity():
    """Page size 1 with last_page_len 1 (the pages' own configuration) maps
    every index to itself."""
    g = torch.Generator().manual_seed(71)
    idx = torch.randint(0, 1 << 20, (500,), generator=g, dtype=torch.int32)
    ptr = torch.tensor([0, 0, 120, 121, 500], dtype=torch.int32)
    tptr, tidx = oracle.expand_paged_kv_indices(ptr, idx, torch.ones(4, dtype=torch.int32), 1)
    assert torch.equal(tptr, ptr) and torch.equal(tidx, idx)


@pytest.mark.parametrize("ps", [2, 16, 64])
def test_paged_indices_are_page_blocks(ps):
    """Random page tables: the slots equal numpy's arange blocks of each page
    (ps consecutive slots per page, the last page cut at last_page_len)."""
    rng = np.random.default_rng(ps)
    bs = 9
    pages = rng.integers(0, 6, size=bs)
    pages[0] = 0
    last = rng.integers(1, ps + 1, size=bs)
    ptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    idx = rng.permutation(1000)[: ptr[-1]].astype(np.int32)
    tptr, tidx = oracle.expand_paged_kv_indices(torch.from_numpy(ptr), torch.from_numpy(idx),
                                                torch.from_numpy(last.astype(np.int32)), ps)
    want = []
    for b in range(bs):
        for k in range(pages[b]):
            n = ps if k < pages[b] - 1 else last[b]
            want.append(idx[ptr[b] + k] * ps + np.arange(n))
    want = np.concatenate(want) if want else np.zeros(0, np.int32)
    assert np.array_equal(tidx.numpy(), want)
    t = np.where(pages > 0, (pages - 1) * ps + last, 0)
    assert np.array_equal(tptr.numpy(), np.concatenate([[0], np.cumsum(t)]))


def test_decode_over_a_paged_pool_equals_decode_over_its_tokens():
    """A pool laid out in pages of 16 (every sequence's tokens in its own
    pages, in order, pages shuffled over the pool): decode through the
    expanded page table equals decode through the tokens' own slots."""
    ps = 16
    wl = W.draw(W.WorkloadSpec("dec", batch=4, hq=8, hkv=2, lq=64, lv=64,
                               prefix=[40, 15, 0, 70], extend=[1, 1, 1, 1], num_slots=1024,
                               seed=72, decode=True))
    g = torch.Generator().manual_seed(73)
    t = [p + 1 for p in wl.prefix_lens]
    n_pages = [(x + ps - 1) // ps for x in t]
    page_ids = torch.randperm(1024 // ps, generator=g)[: sum(n_pages)].to(torch.int32)
    kb_tok, vb_tok = wl.pool()
    kb = torch.zeros_like(kb_tok)
    vb = torch.zeros_like(vb_tok)
    ptr, slots, p0 = [0], [], 0
    for b in range(wl.batch):
        o = int(wl.token_offsets[b])
        for j in range(t[b]):
            s = int(page_ids[p0 + j // ps]) * ps + j % ps
            slots.append(s)
            kb[s] = wl.k_rows[o + j]
            vb[s] = wl.v_rows[o + j]
        p0 += n_pages[b]
        ptr.append(p0)
    last = torch.tensor([x - (n - 1) * ps for x, n in zip(t, n_pages)], dtype=torch.int32)
    tptr, tidx = oracle.expand_paged_kv_indices(torch.tensor(ptr, dtype=torch.int32), page_ids,
                                                last, ps)
    assert tidx.tolist() == slots
    o1, l1 = oracle.decode_attention(wl.q, kb, vb, tptr, tidx, wl.sm_scale)
    o2, l2 = oracle.decode_attention(wl.q, kb_tok, vb_tok, wl.kv_indptr, wl.kv_indices,
                                     wl.sm_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
