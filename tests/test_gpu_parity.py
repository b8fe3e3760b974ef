"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on the same seeded inputs.

Bar: unified indices bit-exact; bf16 attention outputs within max|err| 2e-2
and mean|err| 2e-3, fp32 lse within 1e-3 (tests/gpu_cases.py).
"""
import json
import math
import os

import pytest
import torch

import oracle
from paged_kv_extend_gb300 import pkx
from paged_kv_extend_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_cases import (DEV, DeviceWorkload, assert_close, oracle_decode, oracle_extend,
                           random_masks, sample_rows)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkx.load_library()


# --------------------------------------------------------- unified indices
def _unified_gpu(pptr, pidx, start, elen, eidx, bs, fill=-5):
    d = lambda t: t.to(DEV)
    uptr = torch.full((bs + 1,), fill, dtype=torch.int32, device=DEV)
    uidx = torch.full((pidx.numel() + eidx.numel(),), fill, dtype=torch.int64, device=DEV)
    plen = torch.full((bs,), fill, dtype=torch.int32, device=DEV)
    pkx.build_unified_kv_indices(d(pptr.to(torch.int32)), d(pidx), d(start), d(elen), d(eidx), bs,
                                 out=(uptr, uidx, plen))
    torch.cuda.synchronize()
    return uptr.cpu(), uidx.cpu(), plen.cpu()


def test_unified_indices_hand_fixture_bit_exact():
    fx = json.load(open(os.path.join(GOLDEN, "unified_indices_hand.json")))
    i, e = fx["inputs"], fx["expected"]
    t = lambda k: torch.tensor(i[k], dtype=torch.int32)
    uptr, uidx, plen = _unified_gpu(t("prefix_kv_indptr"), t("prefix_kv_indices"),
                                    t("extend_start_loc"), t("extend_seq_lens"),
                                    t("extend_kv_indices"), i["bs"])
    n = e["unified_kv_indptr"][-1]
    assert uptr.tolist() == e["unified_kv_indptr"]
    assert uidx[:n].tolist() == e["unified_kv_indices_prefix"]
    assert torch.all(uidx[n:] == -5)
    assert plen.tolist() == e["prefix_lens"]


@pytest.mark.parametrize("seed,bs", [(0, 1), (1, 7), (2, 64), (3, 300)])
def test_unified_indices_bit_exact_vs_oracle(seed, bs):
    g = torch.Generator().manual_seed(seed)
    plens = torch.randint(0, 700, (bs,), generator=g)
    plens[torch.rand(bs, generator=g) < 0.2] = 0
    elens = torch.randint(0, 300, (bs,), generator=g).to(torch.int32)
    pptr = torch.zeros(bs + 1, dtype=torch.int32)
    pptr[1:] = torch.cumsum(plens, 0)
    pidx = torch.randint(0, 2**31 - 1, (int(plens.sum()),), generator=g, dtype=torch.int32)
    perm = torch.randperm(bs, generator=g)
    start = torch.zeros(bs, dtype=torch.int32)
    pos = 0
    for b in perm.tolist():
        pos += int(torch.randint(0, 3, (1,), generator=g))
        start[b] = pos
        pos += int(elens[b])
    eidx = torch.randint(0, 2**31 - 1, (pos + 2,), generator=g, dtype=torch.int32)
    uptr, uidx, plen = _unified_gpu(pptr, pidx, start, elens, eidx, bs)
    rptr, ridx, rplen = oracle.build_unified_kv_indices(pptr, pidx, start, elens, eidx, bs, fill=-5)
    assert torch.equal(uptr, rptr)
    assert torch.equal(uidx, ridx)   # includes the untouched tail
    assert torch.equal(plen, rplen)


def test_unified_indices_empty_batch():
    uptr, uidx, plen = _unified_gpu(torch.zeros(1, dtype=torch.int32), torch.zeros(0, dtype=torch.int32),
                                    torch.zeros(0, dtype=torch.int32), torch.zeros(0, dtype=torch.int32),
                                    torch.zeros(0, dtype=torch.int32), 0)
    assert uptr.tolist() == [0]


# ---------------------------------------------------------------- merge_state
@pytest.mark.parametrize("n,h,dv", [(1, 1, 8), (37, 8, 128), (1000, 16, 512), (5, 3, 64)])
def test_merge_state_vs_oracle(n, h, dv):
    g = torch.Generator().manual_seed(n * 31 + dv)
    va = torch.randn(n, h, dv, generator=g).to(torch.bfloat16)
    vb = torch.randn(n, h, dv, generator=g).to(torch.bfloat16)
    sa = torch.randn(n, h, generator=g) * 8
    sb = torch.randn(n, h, generator=g) * 8
    # empty sides
    sa.view(-1)[::7] = float("-inf")
    sb.view(-1)[::11] = float("-inf")
    v, s = pkx.merge_state(va.to(DEV), sa.to(DEV), vb.to(DEV), sb.to(DEV))
    torch.cuda.synchronize()
    rv, rs = oracle.merge_state(va, sa, vb, sb)
    err = (v.double().cpu() - rv).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    fin = torch.isfinite(rs)
    assert torch.equal(torch.isfinite(s.cpu()), fin)
    assert (s.double().cpu()[fin] - rs[fin]).abs().max().item() <= 1e-5 if fin.any() else True


@pytest.mark.parametrize("dv,alias", [(128, "vs"), (512, "vs"), (96, "vs"), (512, "s"),
                                      (96, "v")])
def test_merge_state_in_place(dv, alias):
    """v_out = v_a and / or s_out = s_a.  A 512-dim row spans two warps and a
    96-dim row can span two blocks, so the merged s must not be written
    before every thread of its row has read the inputs."""
    g = torch.Generator().manual_seed(5 + dv)
    n = 300
    va = torch.randn(n, 4, dv, generator=g).to(torch.bfloat16)
    vb = torch.randn(n, 4, dv, generator=g).to(torch.bfloat16)
    sa, sb = torch.randn(n, 4, generator=g) * 4, torch.randn(n, 4, generator=g) * 4
    sa.view(-1)[::13] = float("-inf")
    rv, rs = oracle.merge_state(va, sa, vb, sb)
    a, s_a = va.to(DEV), sa.to(DEV)
    v_out = a if "v" in alias else torch.empty_like(a)
    s_out = s_a if "s" in alias else torch.empty_like(s_a)
    pkx.merge_state(a, s_a, vb.to(DEV), sb.to(DEV), v_out=v_out, s_out=s_out)
    torch.cuda.synchronize()
    err = (v_out.double().cpu() - rv).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert (s_out.double().cpu() - rs).abs().max().item() <= 1e-5


# ------------------------------------------------------------ extend attention
def test_tiny_config():
    """The tiny correctness workload: B=2, Hq=4, Hkv=2, D=64, prefix {16,0},
    extend {8,5}, 64 shuffled slots, scale 1/8."""
    wl = W.draw(W.SPECS["tiny"])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, "tiny")


SMALL = [
    # (lq, hq, hkv, prefix, extend, cap, window)
    (128, 32, 8, [0, 5, 300, 1000], [1, 40, 77, 130], 0.0, -1),
    (128, 32, 8, [17, 0, 2000], [129, 3, 64], 30.0, -1),
    (128, 28, 4, [600, 0, 90, 3000], [200, 1, 19, 5], 0.0, 100),
    (128, 8, 8, [40, 1300], [70, 33], 0.0, -1),
    (128, 16, 1, [250, 7], [9, 260], 5.0, 31),
    (64, 4, 2, [16, 0], [8, 5], 0.0, -1),
    (64, 12, 3, [0, 999, 45], [500, 2, 129], 0.0, 250),
    (64, 64, 4, [128, 1], [16, 256], 12.0, -1),
    (128, 32, 8, [0, 0, 0], [0, 5, 0], 0.0, -1),   # empty sequences around one
]


@pytest.mark.parametrize("lq,hq,hkv,prefix,extend,cap,window", SMALL)
def test_extend_small_vs_oracle(lq, hq, hkv, prefix, extend, cap, window):
    spec = W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lq, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window,
                        seed=sum(prefix) + 3 * sum(extend) + hq)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, f"extend {lq} {hq}/{hkv}")
    # unified form on the same data gives the same answer
    uo, ul, ws2 = dw.unified()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(uo, ul, ro, rl, "unified")


@pytest.mark.parametrize("lq,hq,hkv,prefix,extend,cap,window", SMALL)
def test_ragged_paged_split_vs_oracle(lq, hq, hkv, prefix, extend, cap, window):
    """The ragged + paged + merge_state split gives the two-stage result
    (the oracle's) within the same bar, including sequences without prefix
    (their paged pass is empty) and windows that cut into the prefix."""
    spec = W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lq, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window,
                        seed=sum(prefix) + 3 * sum(extend) + hq)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.ragged_paged()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, f"ragged+paged {lq} {hq}/{hkv}")


def test_ragged_paged_split_mla():
    spec = W.small_spec(batch=3, hq=16, hkv=1, lq=576, lv=512, prefix=[300, 0, 129],
                        extend=[64, 130, 1], sm_scale=1.0 / math.sqrt(192.0), std=0.5,
                        v_aliases_k=True, seed=91)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.ragged_paged()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, "ragged+paged mla")


def test_ragged_paged_split_full_size_sampled_rows():
    """The Llama-3-8B-shaped batch (8353 extend tokens, past the pages' 4096
    threshold for the split) through the split path, sampled rows."""
    wl = W.draw(W.SPECS["llama3_8b"])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.ragged_paged()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, wl.spec.hq, 3072, seed=78)
    ro, rl = oracle_extend(wl, rows=rows)
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, "ragged+paged llama3_8b")
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("scale,cap,window", [
    (-0.09, 0.0, -1),   # negative scale: the row max is scale * min(q.k)
    (0.0, 0.0, -1),     # uniform weights over the visible keys
    (0.6, 0.0, -1),     # large logits: many lazy rescales
    (-0.2, 20.0, 50),   # negative scale through the cap, with a window
])
def test_extend_scale_values(scale, cap, window):
    spec = W.small_spec(batch=3, hq=16, hkv=4, prefix=[0, 260, 1100], extend=[140, 7, 300],
                        logit_cap=cap, sliding_window=window, seed=77)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.unified(scale=scale)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl, scale=scale)
    assert_close(o, lse, ro, rl, f"scale {scale}")


# ------------------------------------------ custom mask and attention sinks
MASK_SINK = [
    # (lq, hq, hkv, prefix, extend, cap, window, mask, sinks)
    (128, 32, 8, [0, 40, 300], [17, 64, 130], 0.0, -1, True, False),
    (128, 32, 8, [900, 5], [70, 200], 0.0, -1, True, False),       # split key ranges
    (128, 16, 4, [33, 260], [9, 40], 0.0, 100, True, False),        # mask and window
    (128, 32, 8, [0, 40, 300], [17, 64, 130], 0.0, -1, False, True),
    (128, 32, 8, [1400, 20], [33, 90], 25.0, -1, False, True),      # sinks, cap, split rows
    (64, 12, 3, [500, 0, 77], [40, 129, 3], 0.0, -1, True, True),
    (128, 28, 4, [700, 64], [100, 5], 0.0, 50, True, True),
]


@pytest.mark.parametrize("lq,hq,hkv,prefix,extend,cap,window,mask,sinks", MASK_SINK)
def test_extend_custom_mask_and_sinks_vs_oracle(lq, hq, hkv, prefix, extend, cap, window,
                                                mask, sinks):
    """Custom mask (replaces the causal mask, keeps the window) and sinks
    (extra denominator term per query head), two-stage and unified forms,
    against the oracle."""
    spec = W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lq, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window,
                        seed=sum(prefix) + 7 * sum(extend) + hq)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    kw = {}
    if mask:
        cm, mi = random_masks(wl, seed=sum(extend))
        kw.update(custom_mask=cm, mask_indptr=mi)
    if sinks:
        g = torch.Generator().manual_seed(hq)
        kw["sinks"] = (torch.randn(hq, generator=g) * 2.0).float()
    ro, rl = oracle_extend(wl, **kw)
    o, lse, ws = dw.extend(**kw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"two-stage mask={mask} sinks={sinks}")
    uo, ul, ws2 = dw.unified(**kw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(uo, ul, ro, rl, f"unified mask={mask} sinks={sinks}")


def test_mask_rows_without_visible_keys_in_a_split_chunk():
    """With a mask a row may see nothing in a split chunk (or nothing at
    all): o = 0 there, lse = -inf, or the sink when one is given."""
    spec = W.small_spec(batch=1, hq=8, hkv=2, lq=128, lv=128, prefix=[1500], extend=[40], seed=3)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    E, P = 40, 1500
    m = torch.zeros(E, P + E, dtype=torch.bool)
    m[:, :64] = True                  # only the first prefix keys ...
    m[5] = False                      # ... and row 5 sees nothing
    flat = m.to(torch.uint8).reshape(-1)
    mi = torch.tensor([0, E * (P + E)], dtype=torch.int32)
    for sinks in (None, torch.linspace(-2.0, 3.0, 8).float()):
        kw = dict(custom_mask=flat, mask_indptr=mi, sinks=sinks)
        ro, rl = oracle_extend(wl, **kw)
        o, lse, ws = dw.unified(**kw)
        torch.cuda.synchronize()
        assert pkx.workspace_status(ws) == 0
        assert_close(o, lse, ro, rl, f"empty rows sinks={sinks is not None}")


@pytest.mark.parametrize("prefix,extend,window,mask,sinks", [
    ([0, 300], [40, 70], -1, True, False),
    ([700, 20], [9, 130], -1, False, True),
    ([150, 2], [60, 17], 40, True, True),
])
def test_mla_custom_mask_and_sinks_vs_oracle(prefix, extend, window, mask, sinks):
    """The MLA head (576/512, V aliases K) with a custom mask and/or sinks,
    two-stage and unified forms."""
    spec = W.small_spec(batch=len(prefix), hq=16, hkv=1, lq=576, lv=512, prefix=prefix,
                        extend=extend, sliding_window=window, std=0.5, v_aliases_k=True,
                        sm_scale=1.0 / math.sqrt(192.0), seed=sum(prefix) + sum(extend))
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    kw = {}
    if mask:
        cm, mi = random_masks(wl, seed=5)
        kw.update(custom_mask=cm, mask_indptr=mi)
    if sinks:
        kw["sinks"] = torch.linspace(-1.0, 2.5, 16).float()
    ro, rl = oracle_extend(wl, **kw)
    o, lse, ws = dw.extend(**kw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"mla two-stage mask={mask} sinks={sinks}")
    uo, ul, ws2 = dw.unified(**kw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(uo, ul, ro, rl, f"mla unified mask={mask} sinks={sinks}")


def test_repeat_calls_are_bitwise_identical():
    wl = W.draw(W.small_spec(batch=3, hq=32, hkv=8, prefix=[700, 30, 0], extend=[90, 300, 17], seed=4))
    dw = DeviceWorkload(wl)
    o1, l1, ws = dw.extend()
    o2, l2, _ = dw.extend()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_no_lse_output_is_fine():
    wl = W.draw(W.small_spec(batch=2, hq=8, hkv=2, prefix=[10, 600], extend=[20, 40], seed=9))
    dw = DeviceWorkload(wl)
    o, _ = dw.out()
    pkx.extend_attention_fwd(dw.q, dw.k_extend, dw.v_extend, o, dw.k_buffer, dw.v_buffer,
                             dw.qo_indptr, dw.kv_indptr, dw.kv_indices, wl.sm_scale)
    torch.cuda.synchronize()
    ro, rl = oracle_extend(wl)
    assert_close(o, rl.float(), ro, rl, "no lse")


# --------------------------------------------------------------------- decode
@pytest.mark.parametrize("lq,hq,hkv,lens,cap,window", [
    (128, 32, 8, [1, 2, 130, 4000, 777], 0.0, -1),
    (128, 32, 8, [300, 1, 9000], 30.0, 64),
    (64, 16, 16, [5, 1000], 0.0, -1),
    (128, 16, 1, [513, 2], 0.0, -1),
])
def test_decode_small_vs_oracle(lq, hq, hkv, lens, cap, window):
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=hq, hkv=hkv, lq=lq, lv=lq,
                          prefix=[x - 1 for x in lens], extend=[1] * len(lens),
                          num_slots=2 * sum(lens) + 16, logit_cap=cap, sliding_window=window,
                          seed=sum(lens), decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, "decode")


def test_decode_padding_sequence_gives_zero():
    """A padded decode slot (T = 0, as CUDA-graph padding produces) yields
    o = 0 and lse = -inf and leaves its neighbours alone."""
    spec = W.WorkloadSpec("dec", batch=3, hq=8, hkv=2, lq=128, lv=128, prefix=[50, 0, 9],
                          extend=[1, 1, 1], num_slots=256, seed=3, decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    kvp = torch.tensor([0, 51, 51, 61], dtype=torch.int32)
    idx = torch.cat([wl.kv_indices[:51], wl.kv_indices[52:62]])
    dw.kv_indptr, dw.kv_indices = kvp.to(DEV), idx.to(DEV)
    o, lse, _ = dw.decode()
    torch.cuda.synchronize()
    kb, vb = wl.pool()
    ro, rl = oracle.decode_attention(wl.q, kb, vb, kvp, idx, wl.sm_scale)
    assert torch.all(o[1].cpu() == 0) and torch.all(torch.isneginf(lse[1].cpu()))
    assert_close(o, lse, ro, rl, "decode padding")


# ------------------------------------------------------------- error paths
def test_out_of_range_index_is_reported_not_dereferenced():
    wl = W.draw(W.small_spec(batch=2, hq=8, hkv=2, prefix=[40, 9], extend=[5, 7], seed=12))
    dw = DeviceWorkload(wl)
    bad = dw.kv_indices.clone()
    bad[3] = wl.spec.num_slots + 1000
    bad[7] = -4
    dw.kv_indices = bad
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == pkx.PKX_EDEVICE
    assert torch.isfinite(o.float()).all()
    # the next good call clears the status word
    dw.kv_indices = wl.kv_indices.to(DEV)
    o, lse, ws = dw.extend()
    assert pkx.workspace_status(ws) == pkx.PKX_OK


def test_workspace_too_small_is_rejected():
    wl = W.draw(W.small_spec(batch=1, hq=8, hkv=2, prefix=[4], extend=[4], seed=1))
    dw = DeviceWorkload(wl)
    o, lse = dw.out()
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkx.PkxError) as e:
        pkx.extend_attention_fwd(dw.q, dw.k_extend, dw.v_extend, o, dw.k_buffer, dw.v_buffer,
                                 dw.qo_indptr, dw.kv_indptr, dw.kv_indices, wl.sm_scale,
                                 lse=lse, workspace=ws)
    assert e.value.code == pkx.PKX_EWORKSPACE


# ------------------------------------------------- full-size sampled parity
@pytest.mark.parametrize("name", ["llama3_8b", "long_prefix", "heavy_tail"])
def test_full_size_sampled_rows(name):
    """The full-size workloads through the two-stage call (prefix from the
    pool, extend rows from k_extend / v_extend); the oracle computes a
    seeded sample of (token, head) rows."""
    wl = W.draw(W.SPECS[name])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, wl.spec.hq, 3072, seed=77)
    ro, rl = oracle_extend(wl, rows=rows)
    hq = wl.spec.hq
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, name)
    assert torch.isfinite(o.float()).all()
    del dw


def _unified_oracle_indices(wl):
    return oracle.build_unified_kv_indices(wl.kv_indptr, wl.kv_indices, wl.extend_start_loc,
                                           wl.extend_seq_lens, wl.extend_kv_indices, wl.batch)


@pytest.mark.parametrize("name", ["llama3_8b", "heavy_tail", "long_prefix", "mla"])
def test_full_size_unified_sampled_rows(name):
    """The benchmarked step itself: build_unified_kv_indices on the GPU, then
    extend_attention_fwd_unified over every key of the pool, at full size
    and in the launch configuration bench.py times.  The GPU-built indices
    are compared bit for bit with the oracle's; the oracle's unified
    attention (over its own indices) computes a seeded sample of 3072
    (token, head) rows."""
    wl = W.draw(W.SPECS[name])
    dw = DeviceWorkload(wl)
    uptr, uidx, plen = pkx.build_unified_kv_indices(
        dw.kv_indptr, dw.kv_indices, dw.extend_start_loc, dw.extend_seq_lens,
        dw.extend_kv_indices, wl.batch)
    rptr, ridx, rplen = _unified_oracle_indices(wl)
    n_u = int(rptr[-1])
    assert torch.equal(uptr.cpu(), rptr) and torch.equal(plen.cpu(), rplen)
    assert torch.equal(uidx.cpu()[:n_u], ridx[:n_u])
    s = wl.spec
    o, lse = dw.out()
    ws = pkx.extend_attention_fwd_unified(dw.q, o, dw.k_buffer, dw.v_buffer, dw.qo_indptr, uptr,
                                          uidx, plen, wl.sm_scale, s.logit_cap, s.sliding_window,
                                          lse=lse)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, s.hq, 3072, seed=79)
    kb, vb = wl.pool()
    ro, rl = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, rptr, ridx, rplen,
                                             wl.sm_scale, s.logit_cap, s.sliding_window,
                                             rows=rows)
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, f"{name} unified")
    assert torch.isfinite(o.float()).all()
    del dw


@pytest.mark.parametrize("name", ["spec_verify", "sinks_swa"])
def test_full_size_mask_and_sinks_sampled_rows(name):
    """The draft-tree verification workload (custom mask) and the sink +
    sliding-window workload at full size, through the unified call the
    benchmark times; the oracle computes a seeded sample of rows."""
    wl = W.draw(W.SPECS[name])
    dw = DeviceWorkload(wl)
    kw = {}
    if wl.custom_mask is not None:
        kw.update(custom_mask=wl.custom_mask, mask_indptr=wl.mask_indptr)
    if wl.sinks is not None:
        kw["sinks"] = wl.sinks.float()
    o, lse, ws = dw.unified(**kw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, wl.spec.hq, 2048, seed=78)
    ro, rl = oracle_extend(wl, rows=rows, **kw)
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, name)
    assert torch.isfinite(o.float()).all()
    del dw


def test_full_size_decode():
    wl = W.draw(W.SPECS["decode_gqa"])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, "decode_gqa")


# ------------------------------------------------------------------ MLA
MLA_SMALL = [
    # (prefix, extend, cap, window)
    ([0, 70, 300], [9, 1, 130], 0.0, -1),
    ([33, 0], [64, 200], 0.0, 50),
    ([129, 5, 2], [17, 40, 3], 20.0, -1),
]


@pytest.mark.parametrize("prefix,extend,cap,window", MLA_SMALL)
def test_mla_small_vs_oracle(prefix, extend, cap, window):
    """MLA head (Lq=576 = 512 latent + 64 rope, Lv=512, V = the first 512
    dims of K, one KV head, 16 query heads)."""
    spec = W.small_spec(batch=len(prefix), hq=16, hkv=1, lq=576, lv=512, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window, std=0.5,
                        v_aliases_k=True, sm_scale=1.0 / math.sqrt(192.0),
                        seed=sum(prefix) + 5 * sum(extend))
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, "mla extend")
    uo, ul, ws2 = dw.unified()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(uo, ul, ro, rl, "mla unified")


def test_mla_decode_small_vs_oracle():
    lens = [1, 64, 65, 1000, 3]
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=16, hkv=1, lq=576, lv=512,
                          prefix=[x - 1 for x in lens], extend=[1] * len(lens),
                          num_slots=4096, sm_scale=1.0 / math.sqrt(192.0), std=0.5,
                          seed=31, v_aliases_k=True, decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, "mla decode")


@pytest.mark.parametrize("hq,lens", [
    # many short sequences around a long one: shares of the key tiles cut
    # through several sequences and split the long one (G = 16)
    (16, [1, 2, 3, 64, 65, 129, 4000, 1, 700, 5] * 3),
    (8, [3000, 1, 1, 1, 300, 64, 2]),        # G = 8
    (32, [5000, 1, 1, 1, 300]),              # G = 32: the largest small-group layout
    (64, [70, 2000, 1, 129]),                # G = 64: the four-stage layout
    (16, [150000]),                          # one sequence over every pair
])
def test_mla_decode_stream_partition_vs_oracle(hq, lens):
    """MLA decode with one KV head splits the key tiles of all sequences laid
    end to end into one equal share per CTA pair."""
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=hq, hkv=1, lq=576, lv=512,
                          prefix=[x - 1 for x in lens], extend=[1] * len(lens),
                          num_slots=sum(lens) + 4096, sm_scale=1.0 / math.sqrt(192.0), std=0.5,
                          seed=sum(lens) % 1000 + hq, v_aliases_k=True, decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, "mla decode, stream partition")


def test_mla_decode_padding_sequence_gives_zero():
    """A padded MLA decode slot (T = 0) yields o = 0 and lse = -inf; its
    neighbours' shares are unaffected."""
    spec = W.WorkloadSpec("dec", batch=3, hq=16, hkv=1, lq=576, lv=512, prefix=[900, 0, 33],
                          extend=[1, 1, 1], num_slots=2048, sm_scale=1.0 / math.sqrt(192.0),
                          std=0.5, seed=4, v_aliases_k=True, decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    kvp = torch.tensor([0, 901, 901, 935], dtype=torch.int32)
    idx = torch.cat([wl.kv_indices[:901], wl.kv_indices[902:936]])
    dw.kv_indptr, dw.kv_indices = kvp.to(DEV), idx.to(DEV)
    o, lse, _ = dw.decode()
    torch.cuda.synchronize()
    kb, vb = wl.pool()
    ro, rl = oracle.decode_attention(wl.q, kb, vb, kvp, idx, wl.sm_scale)
    assert torch.all(o[1].cpu() == 0) and torch.all(torch.isneginf(lse[1].cpu()))
    assert_close(o, lse, ro, rl, "mla decode padding")


def test_mla_requires_v_alias():
    """Lq=576/Lv=512 with a V pool that is not a view of K is refused."""
    spec = W.small_spec(batch=1, hq=16, hkv=1, lq=576, lv=512, prefix=[4], extend=[4],
                        seed=2, v_aliases_k=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    dw.v_buffer = dw.v_buffer.clone()
    o, lse = dw.out()
    with pytest.raises(pkx.PkxError) as e:
        dw.extend()
    assert e.value.code == pkx.PKX_EUNSUPPORTED


@pytest.mark.parametrize("name", ["mla"])
def test_full_size_mla_sampled_rows(name):
    wl = W.draw(W.SPECS[name])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, wl.spec.hq, 2048, seed=78)
    ro, rl = oracle_extend(wl, rows=rows)
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, name)
    assert torch.isfinite(o.float()).all()


def test_full_size_decode_mla():
    wl = W.draw(W.SPECS["decode_mla"])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, "decode_mla")


# ---------------------------------------------------- split head dims
SPLIT_SMALL = [
    # (lq, lv, hq, hkv, prefix, extend, cap, window)
    (192, 128, 16, 16, [0, 70, 300], [9, 1, 130], 0.0, -1),
    (192, 128, 32, 8, [129, 5, 1000], [17, 300, 3], 20.0, -1),
    (192, 128, 16, 2, [33, 0, 700], [64, 200, 1], 0.0, 50),
    (288, 256, 16, 16, [0, 70, 300], [9, 1, 130], 0.0, -1),
    (288, 256, 16, 4, [129, 5, 600], [17, 250, 3], 30.0, 100),
    (288, 256, 8, 1, [0, 257], [300, 40], 0.0, -1),
]


@pytest.mark.parametrize("lq,lv,hq,hkv,prefix,extend,cap,window", SPLIT_SMALL)
def test_split_head_dims_vs_oracle(lq, lv, hq, hkv, prefix, extend, cap, window):
    """The split head dims of the pages' launcher (Lq = 192 = 128 + 64 and
    Lq = 288 = 256 + 32, with Lv = 128 / 256): two-stage and unified extend
    against the oracle over ragged batches with tails, GQA groups, cap and
    window."""
    spec = W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lv, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window,
                        seed=lq + sum(prefix) + 3 * sum(extend))
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    ro, rl = oracle_extend(wl)
    o, lse, ws = dw.extend()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"{lq}/{lv} two-stage")
    uo, ul, ws2 = dw.unified()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(uo, ul, ro, rl, f"{lq}/{lv} unified")


@pytest.mark.parametrize("lq,lv", [(192, 128), (288, 256)])
def test_split_head_dims_decode_vs_oracle(lq, lv):
    lens = [1, 64, 129, 1000, 3, 4097]
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=16, hkv=4, lq=lq, lv=lv,
                          prefix=[x - 1 for x in lens], extend=[1] * len(lens),
                          num_slots=16384, seed=lq + 11, decode=True)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.decode()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ro, rl = oracle_decode(wl)
    assert_close(o, lse, ro, rl, f"{lq}/{lv} decode")


@pytest.mark.parametrize("name", ["split_192", "split_288"])
def test_full_size_split_head_dims_sampled_rows(name):
    """The split-head-dim workloads at full size through the unified call the
    benchmark times (GPU-built indices); 2048 sampled rows against the
    oracle."""
    wl = W.draw(W.SPECS[name])
    dw = DeviceWorkload(wl)
    o, lse, ws = dw.unified()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(wl.n_q_tokens, wl.spec.hq, 2048, seed=81)
    ro, rl = oracle_extend(wl, rows=rows)
    go = o.view(-1, o.shape[-1])[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, name)
    assert torch.isfinite(o.float()).all()


def test_split_head_dims_refuse_mask_and_fp8():
    spec = W.small_spec(batch=1, hq=8, hkv=2, lq=192, lv=128, prefix=[4], extend=[4], seed=3)
    wl = W.draw(spec)
    dw = DeviceWorkload(wl)
    mask, mptr = random_masks(wl, seed=1)
    with pytest.raises(pkx.PkxError) as e:
        dw.extend(custom_mask=mask, mask_indptr=mptr)
    assert e.value.code == pkx.PKX_EUNSUPPORTED
