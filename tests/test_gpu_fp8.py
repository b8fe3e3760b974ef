"""GPU parity over fp8 (e4m3 / e5m2) KV pools: the fp8 KV write bit-exact
against the oracle's codes, and decode / two-stage / unified attention over
an fp8 pool with k_scale / v_scale against the oracle reading the same
codes, within the bf16 bar.  Pools are quantized on the CPU by torch."""
import math

import pytest
import torch

import oracle
from paged_kv_extend_gb300 import pkx
from paged_kv_extend_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_cases import DEV, assert_close, sample_rows

FMTS = [torch.float8_e4m3fn, torch.float8_e5m2]


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkx.load_library()


def _as_codes(t):
    return t.cpu().view(torch.uint8)


# ------------------------------------------------------------ fp8 KV write
@pytest.mark.parametrize("dt", FMTS)
@pytest.mark.parametrize("n,hkv,d,ks,vs,amp", [
    (1, 1, 64, 1.0, 1.0, 1.0), (77, 8, 128, 0.37, 2.5, 3.0), (300, 2, 64, 1.0, 1.0, 1e-3),
    (129, 4, 128, 1.0, 1.0, 600.0)])
def test_fp8_write_bit_exact(dt, n, hkv, d, ks, vs, amp):
    """Codes bit-exact against the oracle: non-power-of-two scales, values in
    the subnormal range, values that saturate, strided inputs."""
    g = torch.Generator().manual_seed(n + d)
    slots = 2 * n + 5
    kb = torch.randint(0, 120, (slots, hkv, d), generator=g, dtype=torch.uint8).view(dt)
    vb = torch.randint(0, 120, (slots, hkv, d), generator=g, dtype=torch.uint8).view(dt)
    loc = torch.randperm(slots, generator=g)[:n]
    k = (torch.randn(n, hkv + 1, d, generator=g) * amp).to(torch.bfloat16)[:, 1:]
    v = (torch.randn(n, hkv, d, generator=g) * amp).to(torch.bfloat16)
    k[0, 0, :4] = torch.tensor([0.0, -0.0, 1e-30, -1e-30])
    want_k, want_v = oracle.set_kv_buffer_fp8(kb, vb, loc, k, v, ks, vs)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    pkx.set_kv_buffer_fp8(dkb, dvb, loc.to(DEV), k.to(DEV), v.to(DEV), ks, vs)
    torch.cuda.synchronize()
    assert torch.equal(_as_codes(dkb), _as_codes(want_k))
    assert torch.equal(_as_codes(dvb), _as_codes(want_v))


# ------------------------------------------------------- attention over fp8
def _extend_case(dt, lq, hq, hkv, prefix, extend, cap, window, ks, vs, seed):
    lv = {192: 128, 288: 256}.get(lq, lq)  # the split head dims
    spec = W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lv, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window, seed=seed)
    wl = W.draw(spec)
    kb, vb = wl.pool_fp8(dt, ks, vs)
    return wl, kb, vb


CASES = [
    # (lq, hq, hkv, prefix, extend, cap, window, k_scale, v_scale)
    (128, 32, 8, [0, 5, 300, 1000], [1, 40, 77, 130], 0.0, -1, 1.0, 1.0),
    (128, 28, 4, [600, 0, 90, 3000], [200, 1, 19, 5], 20.0, 100, 0.05, 0.02),
    (64, 12, 3, [0, 999, 45], [500, 2, 129], 0.0, 250, 0.5, 2.0),
    (64, 8, 8, [40, 1300], [70, 33], 5.0, -1, 0.25, 0.125),
    # the split head dims (one Q tile per unit)
    (192, 16, 16, [0, 70, 300], [9, 1, 130], 0.0, -1, 0.5, 0.25),
    (192, 32, 8, [129, 5, 1000], [17, 300, 3], 20.0, 100, 0.05, 0.02),
    (288, 16, 1, [0, 2000, 33], [64, 1, 200], 0.0, -1, 1.0, 2.0),
    (288, 8, 2, [500, 7], [3, 150], 5.0, 64, 0.25, 0.125),
]


@pytest.mark.parametrize("dt", FMTS)
@pytest.mark.parametrize("lq,hq,hkv,prefix,extend,cap,window,ks,vs", CASES)
def test_extend_over_fp8_pool(dt, lq, hq, hkv, prefix, extend, cap, window, ks, vs):
    """Two-stage (fp8 prefix tiles, bf16 extend tiles) and unified (every
    key from the fp8 pool) against the oracle reading the same codes."""
    wl, kb, vb = _extend_case(dt, lq, hq, hkv, prefix, extend, cap, window, ks, vs,
                              seed=sum(prefix) + 7 * sum(extend))
    s = wl.spec
    k_ext, v_ext = wl.extend_kv()
    ro, rl = oracle.extend_attention(wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr,
                                     wl.kv_indices, wl.sm_scale, cap, window,
                                     k_scale=ks, v_scale=vs)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    n = wl.n_q_tokens
    o = torch.full((n, hq, s.lv), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n, hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.extend_attention_fwd(wl.q.to(DEV), k_ext.to(DEV), v_ext.to(DEV), o, dkb, dvb,
                                  wl.qo_indptr.to(DEV), wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, cap, window, lse=lse,
                                  k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"two-stage fp8 {dt}")
    # unified: the extend tokens' K/V must be in the pool as fp8 as well
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    uo, ul = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, cap, window, k_scale=ks, v_scale=vs)
    o2 = torch.full_like(o, float("nan"))
    l2 = torch.full_like(lse, float("nan"))
    ws2 = pkx.extend_attention_fwd_unified(wl.q.to(DEV), o2, dkb, dvb, wl.qo_indptr.to(DEV),
                                           uptr.to(DEV), uidx.to(DEV), plen.to(DEV),
                                           wl.sm_scale, cap, window, lse=l2, k_scale=ks,
                                           v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(o2, l2, uo, ul, f"unified fp8 {dt}")


MASKED = [
    # (lq, hq, hkv, prefix, extend, cap, window, k_scale, v_scale, sinks)
    (128, 32, 8, [0, 40, 300], [17, 64, 130], 0.0, -1, 0.5, 0.25, False),
    (128, 16, 4, [900, 5], [70, 200], 20.0, 100, 0.05, 0.02, True),   # split rows, cap, window
    (64, 12, 3, [500, 0, 77], [40, 129, 3], 0.0, -1, 1.0, 2.0, True),
]


@pytest.mark.parametrize("dt", FMTS)
@pytest.mark.parametrize("lq,hq,hkv,prefix,extend,cap,window,ks,vs,sinks", MASKED)
def test_masked_extend_over_fp8_pool(dt, lq, hq, hkv, prefix, extend, cap, window, ks, vs, sinks):
    """A custom mask (and sinks) over an fp8 pool, two-stage and unified,
    against the oracle reading the same codes with the same mask."""
    from gpu_cases import random_masks
    wl, kb, vb = _extend_case(dt, lq, hq, hkv, prefix, extend, cap, window, ks, vs,
                              seed=3 * sum(prefix) + sum(extend) + hq)
    cm, mi = random_masks(wl, seed=sum(extend) + lq)
    sk = (torch.randn(hq, generator=torch.Generator().manual_seed(hq)) * 2.0).float() \
        if sinks else None
    k_ext, v_ext = wl.extend_kv()
    ro, rl = oracle.extend_attention(wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr,
                                     wl.kv_indices, wl.sm_scale, cap, window, custom_mask=cm,
                                     mask_indptr=mi, sinks=sk, k_scale=ks, v_scale=vs)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    dsk = sk.to(DEV) if sk is not None else None
    n = wl.n_q_tokens
    o = torch.full((n, hq, lq), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n, hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.extend_attention_fwd(wl.q.to(DEV), k_ext.to(DEV), v_ext.to(DEV), o, dkb, dvb,
                                  wl.qo_indptr.to(DEV), wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, cap, window, lse=lse,
                                  custom_mask=cm.to(DEV), mask_indptr=mi.to(DEV), sinks=dsk,
                                  k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"two-stage masked fp8 {dt}")
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    uo, ul = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, cap, window, custom_mask=cm,
                                             mask_indptr=mi, sinks=sk, k_scale=ks, v_scale=vs)
    o2 = torch.full_like(o, float("nan"))
    l2 = torch.full_like(lse, float("nan"))
    ws2 = pkx.extend_attention_fwd_unified(wl.q.to(DEV), o2, dkb, dvb, wl.qo_indptr.to(DEV),
                                           uptr.to(DEV), uidx.to(DEV), plen.to(DEV),
                                           wl.sm_scale, cap, window, lse=l2,
                                           custom_mask=cm.to(DEV), mask_indptr=mi.to(DEV),
                                           sinks=dsk, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(o2, l2, uo, ul, f"unified masked fp8 {dt}")


MLA8 = [
    # (prefix, extend, cap, window, k_scale, v_scale, mask, sinks)
    ([0, 70, 300], [9, 1, 130], 0.0, -1, 0.25, 0.25, False, False),
    ([129, 5], [17, 40], 20.0, 50, 0.5, 0.125, False, False),
    ([60, 300], [33, 70], 0.0, -1, 0.25, 0.25, True, True),
]


@pytest.mark.parametrize("dt", FMTS)
@pytest.mark.parametrize("prefix,extend,cap,window,ks,vs,mask,sinks", MLA8)
def test_mla_extend_over_fp8_pool(dt, prefix, extend, cap, window, ks, vs, mask, sinks):
    """The MLA head (576 / 512, v_buffer a view of k_buffer's codes) over an
    fp8 pool on CTA pairs, two-stage and unified, against the oracle reading
    the same codes (a key reads code * k_scale, a value code * v_scale)."""
    from gpu_cases import random_masks
    spec = W.small_spec(batch=len(prefix), hq=16, hkv=1, lq=576, lv=512, prefix=prefix,
                        extend=extend, logit_cap=cap, sliding_window=window, std=0.5,
                        v_aliases_k=True, sm_scale=1.0 / math.sqrt(192.0),
                        seed=sum(prefix) + 3 * sum(extend))
    wl = W.draw(spec)
    kb, vb = wl.pool_fp8(dt, ks, vs)
    kw = {}
    if mask:
        cm, mi = random_masks(wl, seed=sum(prefix))
        kw.update(custom_mask=cm, mask_indptr=mi)
    if sinks:
        kw["sinks"] = (torch.randn(16, generator=torch.Generator().manual_seed(16)) * 2.0).float()
    dkw = {k: v.to(DEV) for k, v in kw.items()}
    k_ext, v_ext = wl.extend_kv()
    ro, rl = oracle.extend_attention(wl.q, k_ext, v_ext, kb, vb, wl.qo_indptr, wl.kv_indptr,
                                     wl.kv_indices, wl.sm_scale, cap, window, k_scale=ks,
                                     v_scale=vs, **kw)
    dkb = kb.to(DEV)
    dvb = dkb[..., :512]
    dke = k_ext.to(DEV)
    n = wl.n_q_tokens
    o = torch.full((n, 16, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n, 16), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.extend_attention_fwd(wl.q.to(DEV), dke, dke[..., :512], o, dkb, dvb,
                                  wl.qo_indptr.to(DEV), wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, cap, window, lse=lse,
                                  k_scale=ks, v_scale=vs, **dkw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"mla two-stage fp8 {dt}")
    uptr, uidx, plen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    uo, ul = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, uptr, uidx, plen,
                                             wl.sm_scale, cap, window, k_scale=ks, v_scale=vs,
                                             **kw)
    o2 = torch.full_like(o, float("nan"))
    l2 = torch.full_like(lse, float("nan"))
    ws2 = pkx.extend_attention_fwd_unified(wl.q.to(DEV), o2, dkb, dvb, wl.qo_indptr.to(DEV),
                                           uptr.to(DEV), uidx.to(DEV), plen.to(DEV),
                                           wl.sm_scale, cap, window, lse=l2, k_scale=ks,
                                           v_scale=vs, **dkw)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == 0
    assert_close(o2, l2, uo, ul, f"mla unified fp8 {dt}")


@pytest.mark.parametrize("dt", FMTS)
def test_mla_decode_over_fp8_pool(dt):
    lens = [1, 64, 65, 700, 4096]
    spec = W.WorkloadSpec("dec_mla8", batch=len(lens), hq=16, hkv=1, lq=576, lv=512,
                          prefix=[t - 1 for t in lens], extend=[1] * len(lens),
                          num_slots=2 * sum(lens) + 16, sm_scale=1.0 / math.sqrt(192.0),
                          std=0.5, seed=sum(lens), v_aliases_k=True, decode=True)
    wl = W.draw(spec)
    kb, vb = wl.pool_fp8(dt, 0.25, 0.25)
    ro, rl = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     k_scale=0.25, v_scale=0.25)
    dkb = kb.to(DEV)
    o = torch.full((wl.batch, 16, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((wl.batch, 16), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.decode_attention_fwd(wl.q.to(DEV), o, dkb, dkb[..., :512], wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, lse=lse, k_scale=0.25,
                                  v_scale=0.25)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"mla decode fp8 {dt}")


@pytest.mark.parametrize("dt", FMTS)
@pytest.mark.parametrize("lq,hq,hkv,lens,cap,window,ks,vs", [
    (128, 32, 8, [1, 17, 128, 129, 4000], 0.0, -1, 1.0, 1.0),
    (128, 16, 2, [700, 3, 2049], 30.0, 255, 0.1, 0.04),
    (64, 8, 1, [64, 1000, 0], 0.0, -1, 0.5, 4.0)])
def test_decode_over_fp8_pool(dt, lq, hq, hkv, lens, cap, window, ks, vs):
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=hq, hkv=hkv, lq=lq, lv=lq,
                          prefix=[max(t - 1, 0) for t in lens], extend=[1 if t else 0 for t in lens],
                          num_slots=2 * sum(lens) + 16, logit_cap=cap, sliding_window=window,
                          seed=sum(lens), decode=True)
    wl = W.draw(spec)
    kb, vb = wl.pool_fp8(dt, ks, vs)
    ro, rl = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     cap, window, k_scale=ks, v_scale=vs)
    o = torch.full((wl.batch, hq, lq), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.decode_attention_fwd(wl.q.to(DEV), o, kb.to(DEV), vb.to(DEV), wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, cap, window, lse=lse,
                                  k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, f"decode fp8 {dt}")


def test_full_size_decode_over_fp8_pool():
    """The 64 x 8193-key decode batch over an e4m3 pool, every row."""
    wl = W.draw(W.SPECS["decode_gqa"])
    s = wl.spec
    kb, vb = wl.pool_fp8(torch.float8_e4m3fn, 0.0625, 0.0625)
    ro, rl = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     k_scale=0.0625, v_scale=0.0625)
    o = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(s.batch, s.hq, dtype=torch.float32, device=DEV)
    ws = pkx.decode_attention_fwd(wl.q.to(DEV), o, kb.to(DEV), vb.to(DEV), wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, lse=lse, k_scale=0.0625,
                                  v_scale=0.0625)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert_close(o, lse, ro, rl, "decode_gqa fp8")


@pytest.mark.parametrize("name", ["llama3_8b", "long_prefix"])
def test_full_size_unified_extend_over_fp8_pool(name):
    """The benchmarked unified step over an e4m3 pool (k_scale = v_scale =
    0.5, as bench.py's fp8 components): GPU-built unified indices, then the
    unified call; a seeded sample of 3072 rows against the oracle reading the
    same codes through its own unified indices."""
    wl = W.draw(W.SPECS[name])
    s = wl.spec
    ks = vs = 0.5
    kb, vb = wl.pool_fp8(torch.float8_e4m3fn, ks, vs)
    uptr, uidx, plen = pkx.build_unified_kv_indices(
        wl.kv_indptr.to(DEV), wl.kv_indices.to(DEV), wl.extend_start_loc.to(DEV),
        wl.extend_seq_lens.to(DEV), wl.extend_kv_indices.to(DEV), wl.batch)
    rptr, ridx, rplen = oracle.build_unified_kv_indices(
        wl.kv_indptr, wl.kv_indices, wl.extend_start_loc, wl.extend_seq_lens,
        wl.extend_kv_indices, wl.batch)
    n = wl.n_q_tokens
    o = torch.full((n, s.hq, s.lv), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n, s.hq), float("nan"), dtype=torch.float32, device=DEV)
    ws = pkx.extend_attention_fwd_unified(wl.q.to(DEV), o, kb.to(DEV), vb.to(DEV),
                                          wl.qo_indptr.to(DEV), uptr, uidx, plen, wl.sm_scale,
                                          s.logit_cap, s.sliding_window, lse=lse, k_scale=ks,
                                          v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    rows = sample_rows(n, s.hq, 3072, seed=80)
    ro, rl = oracle.extend_attention_unified(wl.q, kb, vb, wl.qo_indptr, rptr, ridx, rplen,
                                             wl.sm_scale, s.logit_cap, s.sliding_window,
                                             rows=rows, k_scale=ks, v_scale=vs)
    go = o.view(-1, s.lv)[rows.to(DEV)]
    gl = lse.view(-1)[rows.to(DEV)]
    assert_close(go, gl, ro, rl, f"{name} unified fp8")
    assert torch.isfinite(o.float()).all()


def test_fp8_write_then_decode_chain():
    """The decode step's own chain on the GPU: the new tokens' K/V written
    into an e5m2 pool by the fp8 KV write, then decode; against the oracle's
    write and decode."""
    wl = W.draw(W.WorkloadSpec("dec", batch=6, hq=16, hkv=4, lq=128, lv=128,
                               prefix=("uniform", 1, 900), extend=("const", 1), num_slots=20000,
                               seed=64, decode=True))
    dt, ks, vs = torch.float8_e5m2, 0.3, 0.7
    kb, vb = wl.pool_fp8(dt, ks, vs)
    last = wl.token_offsets[1:] - 1
    loc = wl.slots[last].to(torch.int64)
    kb.view(torch.uint8)[loc] = 0
    vb.view(torch.uint8)[loc] = 0
    k_new, v_new = wl.k_rows[last], wl.v_rows[last]
    wk, wv = oracle.set_kv_buffer_fp8(kb, vb, loc, k_new, v_new, ks, vs)
    ro, rl = oracle.decode_attention(wl.q, wk, wv, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     k_scale=ks, v_scale=vs)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    pkx.set_kv_buffer_fp8(dkb, dvb, loc.to(DEV), k_new.to(DEV), v_new.to(DEV), ks, vs)
    o = torch.empty(wl.batch, 16, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(wl.batch, 16, dtype=torch.float32, device=DEV)
    ws = pkx.decode_attention_fwd(wl.q.to(DEV), o, dkb, dvb, wl.kv_indptr.to(DEV),
                                  wl.kv_indices.to(DEV), wl.sm_scale, lse=lse, k_scale=ks,
                                  v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert torch.equal(_as_codes(dkb), _as_codes(wk))
    assert_close(o, lse, ro, rl, "write + decode fp8")
