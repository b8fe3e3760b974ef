"""GPU parity of the KV write into the pool (pkx_set_kv_buffer) and the
KV-index gather from the request-to-token table (pkx_create_kv_indices),
called through the C ABI, against the oracle.  Both are integer / byte work:
the bar is bit-exact.
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
    from gpu_cases import DEV, assert_close, oracle_decode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkx.load_library()


def _i64(x):
    return torch.as_tensor(x, dtype=torch.int64).to(DEV) if x is not None else None


def _gather_gpu(table, rpi, lens, start=None, capacity=None, fill=-7):
    table = torch.as_tensor(table, dtype=torch.int32).to(DEV)
    bs = len(rpi)
    total = int(torch.as_tensor(lens).sum()) if bs else 0
    cap = total if capacity is None else capacity
    kvp = torch.full((bs + 1,), fill, dtype=torch.int32, device=DEV)
    kvi = torch.full((cap + 5,), fill, dtype=torch.int32, device=DEV)
    pkx.create_kv_indices(table, _i64(rpi), _i64(lens), _i64(start), kv_indptr=kvp,
                          kv_indices=kvi[:cap])
    torch.cuda.synchronize()
    return kvp.cpu(), kvi.cpu()


# ------------------------------------------------------------ index gather
def test_gather_hand_fixture_bit_exact():
    fx = json.load(open(os.path.join(GOLDEN, "kv_indices_hand.json")))
    for name, c in fx["cases"].items():
        kvp, kvi = _gather_gpu(fx["req_to_token"], c["req_pool_indices"],
                               c["paged_kernel_lens"], c["kv_start_idx"])
        n = c["expected_kv_indptr"][-1]
        assert kvp.tolist() == c["expected_kv_indptr"], name
        assert kvi[:n].tolist() == c["expected_kv_indices"], name
        assert torch.all(kvi[n:] == -7), name


@pytest.mark.parametrize("seed,bs,rows,cols,maxlen,with_start", [
    (0, 1, 2, 64, 64, False), (1, 7, 16, 600, 512, True), (2, 64, 80, 3000, 2900, False),
    (3, 300, 512, 5000, 4000, True), (4, 4096, 4100, 700, 600, True),
    (5, 12000, 12300, 40, 40, False)])
def test_gather_bit_exact_vs_oracle(seed, bs, rows, cols, maxlen, with_start):
    """Random tables, empty and one-entry sequences, lengths that straddle the
    CTA shares, and the largest batch the call takes."""
    g = torch.Generator().manual_seed(seed)
    table = torch.randint(0, 1 << 30, (rows, cols), generator=g, dtype=torch.int32)
    rpi = torch.randperm(rows, generator=g)[:bs]
    lens = torch.randint(0, maxlen + 1, (bs,), generator=g)
    lens[: min(bs, 3)] = torch.tensor([0, 1, maxlen])[: min(bs, 3)]
    start = torch.randint(0, cols - maxlen + 1, (bs,), generator=g) if with_start else None
    want_p, want_i = oracle.create_kv_indices(table, rpi, lens, start)
    kvp, kvi = _gather_gpu(table, rpi, lens, start)
    n = int(want_p[-1])
    assert torch.equal(kvp, want_p)
    assert torch.equal(kvi[:n], want_i)
    assert torch.all(kvi[n:] == -7)


def test_gather_full_size_long_sequences():
    """Sequences of up to 128K tokens (the long-prefix shape) in one call:
    every entry bit-exact against the oracle."""
    g = torch.Generator().manual_seed(11)
    bs, cols = 16, 131072
    table = torch.randint(0, 1 << 22, (bs + 1, cols), generator=g, dtype=torch.int32)
    rpi = torch.arange(1, bs + 1)
    lens = torch.randint(60000, cols + 1, (bs,), generator=g)
    want_p, want_i = oracle.create_kv_indices(table, rpi, lens)
    kvp, kvi = _gather_gpu(table, rpi, lens)
    assert torch.equal(kvp, want_p)
    assert torch.equal(kvi[: int(want_p[-1])], want_i)


def test_gather_respects_capacity_and_table_bounds():
    """Entries past the output capacity are not written; an entry whose
    source lies outside the table reads as -1 (nothing outside the table is
    dereferenced)."""
    table = torch.arange(40, dtype=torch.int32).view(4, 10)
    kvp, kvi = _gather_gpu(table, [1, 2], [6, 6], capacity=8)
    assert kvp.tolist() == [0, 6, 12]
    assert kvi[:8].tolist() == [10, 11, 12, 13, 14, 15, 20, 21]
    assert torch.all(kvi[8:] == -7)
    # row 7 does not exist; columns 8.. of row 3 run off the end of the row
    kvp, kvi = _gather_gpu(table, [7, 3], [2, 4], start=[0, 8])
    assert kvp.tolist() == [0, 2, 6]
    assert kvi[:6].tolist() == [-1, -1, 38, 39, -1, -1]


def test_gather_empty_batch():
    kvp = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    kvi = torch.empty(0, dtype=torch.int32, device=DEV)
    e = torch.empty(0, dtype=torch.int64, device=DEV)
    pkx.create_kv_indices(torch.zeros(2, 4, dtype=torch.int32, device=DEV), e, e, None,
                          kv_indptr=kvp, kv_indices=kvi)
    torch.cuda.synchronize()
    assert kvp.tolist() == [0]


# ------------------------------------------------------------ KV write
def _pools(slots, hkv, lk, lv, seed):
    g = torch.Generator().manual_seed(seed)
    kb = torch.randn(slots, hkv, lk, generator=g).to(torch.bfloat16)
    vb = torch.randn(slots, hkv, lv, generator=g).to(torch.bfloat16)
    return kb, vb, g


@pytest.mark.parametrize("n,hkv,lk,lv,slots,strided", [
    (1, 1, 64, 64, 8, False), (37, 8, 128, 128, 500, False), (300, 2, 64, 64, 4096, True),
    (1000, 4, 128, 96, 3000, True), (129, 3, 8, 16, 400, False)])
def test_kv_write_bit_exact_vs_oracle(n, hkv, lk, lv, slots, strided):
    kb, vb, g = _pools(slots, hkv, lk, lv, n)
    loc = torch.randperm(slots, generator=g)[:n]
    if strided:  # every head row taken out of a wider tensor
        k = torch.randn(n, hkv + 1, lk + 16, generator=g).to(torch.bfloat16)[:, 1:, 16:]
        v = torch.randn(n, hkv, 2 * lv, generator=g).to(torch.bfloat16)[:, :, :lv]
    else:
        k = torch.randn(n, hkv, lk, generator=g).to(torch.bfloat16)
        v = torch.randn(n, hkv, lv, generator=g).to(torch.bfloat16)
    want_k, want_v = oracle.set_kv_buffer(kb, vb, loc, k, v)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    pkx.set_kv_buffer(dkb, dvb, loc.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(dkb.cpu().view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(dvb.cpu().view(torch.int16), want_v.view(torch.int16))


def test_kv_write_k_only_mla_pool():
    """MLA: the pool row is the 576-dim latent; V is its first 512 dims, so
    only K is written."""
    slots, n = 2000, 321
    kb, _, g = _pools(slots, 1, 576, 8, 5)
    loc = torch.randperm(slots, generator=g)[:n]
    k = torch.randn(n, 1, 576, generator=g).to(torch.bfloat16)
    want_k, _ = oracle.set_kv_buffer(kb, kb[..., :512], loc, k, None)
    dkb = kb.to(DEV)
    pkx.set_kv_buffer(dkb, dkb[..., :512], loc.to(DEV), k.to(DEV), None)
    torch.cuda.synchronize()
    assert torch.equal(dkb.cpu().view(torch.int16), want_k.view(torch.int16))


def test_kv_write_skips_slots_outside_the_pool():
    slots = 64
    kb, vb, g = _pools(slots, 2, 64, 64, 6)
    loc = torch.tensor([3, -1, 64, 10, 1 << 40])
    k = torch.randn(5, 2, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(5, 2, 64, generator=g).to(torch.bfloat16)
    dkb, dvb = kb.to(DEV), vb.to(DEV)
    pkx.set_kv_buffer(dkb, dvb, loc.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    keep = torch.tensor([0, 3])
    want_k, want_v = oracle.set_kv_buffer(kb, vb, loc[keep], k[keep], v[keep])
    assert torch.equal(dkb.cpu().view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(dvb.cpu().view(torch.int16), want_v.view(torch.int16))


@pytest.mark.parametrize("name", ["llama3_8b", "mla"])
def test_kv_write_full_size(name):
    """The extend tokens of a full-size workload written into a pool whose
    extend slots hold stale rows: every written row equals its input row
    (any size), and the pool's other rows are untouched."""
    wl = W.draw(W.SPECS[name])
    s = wl.spec
    kb, vb = wl.pool(DEV)
    loc = wl.extend_kv_indices.to(DEV, torch.int64)
    k_ext, v_ext = wl.extend_kv(DEV)
    kb.index_fill_(0, loc, 0.5)
    before = kb.clone()
    if s.v_aliases_k:
        pkx.set_kv_buffer(kb, vb, loc, k_ext, None)
    else:
        vb.index_fill_(0, loc, 0.5)
        pkx.set_kv_buffer(kb, vb, loc, k_ext, v_ext)
        assert torch.equal(vb.index_select(0, loc).view(torch.int16), v_ext.view(torch.int16))
    torch.cuda.synchronize()
    assert torch.equal(kb.index_select(0, loc).view(torch.int16), k_ext.view(torch.int16))
    other = torch.ones(s.num_slots, dtype=torch.bool, device=DEV)
    other[loc] = False
    assert torch.equal(kb[other].view(torch.int16), before[other].view(torch.int16))


# ------------------------------------------ gather + write + attention chain
def test_window_decode_through_gather_matches_windowed_oracle():
    """The sliding-window decode updater's chain on the GPU: the new token's
    K/V written at its slot, the last W+1 slots gathered from the
    request-to-token table, plain decode over them; against windowed decode
    of the oracle over all slots."""
    wl = W.draw(W.WorkloadSpec("dec", batch=24, hq=16, hkv=4, lq=128, lv=128,
                               prefix=("uniform", 1, 3000), extend=("const", 1), num_slots=200000,
                               seed=12, decode=True))
    table, rpi, seq = wl.req_to_token(seed=8)
    Wn = 255
    kb, vb = wl.pool()
    last = (wl.token_offsets[1:] - 1)              # each sequence's new token
    loc = wl.slots[last].to(torch.int64)
    stale_k, stale_v = kb.clone(), vb.clone()
    stale_k[loc] = 0
    stale_v[loc] = 0
    dkb, dvb = stale_k.to(DEV), stale_v.to(DEV)
    pkx.set_kv_buffer(dkb, dvb, loc.to(DEV), wl.k_rows[last].to(DEV), wl.v_rows[last].to(DEV))
    paged = torch.clamp(seq, max=Wn + 1)
    kvp, kvi = pkx.create_kv_indices(table.to(DEV), rpi.to(DEV), paged.to(DEV),
                                     (seq - paged).to(DEV), capacity=int(paged.sum()))
    s = wl.spec
    o = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(s.batch, s.hq, dtype=torch.float32, device=DEV)
    pkx.decode_attention_fwd(wl.q.to(DEV), o, dkb, dvb, kvp, kvi, wl.sm_scale, lse=lse)
    torch.cuda.synchronize()
    want_o, want_l = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices,
                                             wl.sm_scale, sliding_window=Wn)
    assert_close(o.cpu(), lse.cpu(), want_o, want_l)


# ------------------------------------------------------ page tables (page size > 1)
def _expand_gpu(ptr, idx, last, ps, capacity=None, fill=-7):
    ptr = torch.as_tensor(ptr, dtype=torch.int32)
    idx = torch.as_tensor(idx, dtype=torch.int32)
    last = torch.as_tensor(last, dtype=torch.int32)
    want_p, want_i = oracle.expand_paged_kv_indices(ptr, idx, last, ps)
    cap = want_i.numel() if capacity is None else capacity
    tptr = torch.full((ptr.numel(),), fill, dtype=torch.int32, device=DEV)
    tidx = torch.full((cap + 5,), fill, dtype=torch.int32, device=DEV)
    pkx.expand_paged_kv_indices(ptr.to(DEV), idx.to(DEV), last.to(DEV), ps,
                                token_indptr=tptr, token_indices=tidx[:cap])
    torch.cuda.synchronize()
    return tptr.cpu(), tidx.cpu(), want_p, want_i


def test_paged_expansion_hand_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "paged_indices_hand.json")))
    tptr, tidx, _, _ = _expand_gpu(fx["kv_indptr"], fx["kv_indices"], fx["kv_last_page_len"],
                                   fx["page_size"])
    n = fx["expected_token_indptr"][-1]
    assert tptr.tolist() == fx["expected_token_indptr"]
    assert tidx[:n].tolist() == fx["expected_token_indices"]
    assert torch.all(tidx[n:] == -7)


@pytest.mark.parametrize("seed,bs,ps,max_pages", [
    (0, 1, 16, 3), (1, 64, 16, 300), (2, 300, 64, 40), (3, 4096, 8, 20), (4, 12000, 32, 2),
    (5, 16, 128, 1100)])
def test_paged_expansion_bit_exact_vs_oracle(seed, bs, ps, max_pages):
    g = torch.Generator().manual_seed(seed)
    pages = torch.randint(0, max_pages + 1, (bs,), generator=g)
    pages[0] = 0
    ptr = torch.cat([torch.zeros(1, dtype=torch.int64), pages.cumsum(0)])
    idx = torch.randint(0, 1 << 24, (int(ptr[-1]),), generator=g, dtype=torch.int32)
    last = torch.randint(1, ps + 1, (bs,), generator=g)
    tptr, tidx, want_p, want_i = _expand_gpu(ptr, idx, last, ps)
    assert torch.equal(tptr, want_p)
    assert torch.equal(tidx[: want_i.numel()], want_i)


def test_paged_expansion_bounds():
    """A last page longer than the page size reads no page past the
    sequence's own (those keys come out as -1); no entry past the capacity
    is written."""
    tptr, tidx, _, _ = _expand_gpu([0, 1, 2], [3, 5], [6, 2], 4, capacity=7)
    assert tptr.tolist() == [0, 6, 8]
    assert tidx[:7].tolist() == [12, 13, 14, 15, -1, -1, 20]
    assert torch.all(tidx[7:] == -7)


def test_decode_through_a_page_table():
    """Decode over a pool laid out in pages of 16: the page table expanded on
    the GPU, then decode; against the oracle's decode over the tokens' own
    slots."""
    ps = 16
    wl = W.draw(W.WorkloadSpec("dec", batch=12, hq=32, hkv=8, lq=128, lv=128,
                               prefix=("uniform", 0, 2000), extend=("const", 1),
                               num_slots=1 << 16, seed=74, decode=True))
    g = torch.Generator().manual_seed(75)
    t = [p + 1 for p in wl.prefix_lens]
    n_pages = [(x + ps - 1) // ps for x in t]
    page_ids = torch.randperm((1 << 16) // ps, generator=g)[: sum(n_pages)].to(torch.int32)
    kb = torch.zeros(1 << 16, 8, 128, dtype=torch.bfloat16)
    vb = torch.zeros_like(kb)
    ptr, p0 = [0], 0
    for b in range(wl.batch):
        o = int(wl.token_offsets[b])
        slots = page_ids[p0 + torch.arange(t[b]) // ps].long() * ps + torch.arange(t[b]) % ps
        kb[slots] = wl.k_rows[o:o + t[b]]
        vb[slots] = wl.v_rows[o:o + t[b]]
        p0 += n_pages[b]
        ptr.append(p0)
    last = torch.tensor([x - (n - 1) * ps for x, n in zip(t, n_pages)], dtype=torch.int32)
    kvp, kvi = pkx.expand_paged_kv_indices(torch.tensor(ptr, dtype=torch.int32).to(DEV),
                                           page_ids.to(DEV), last.to(DEV), ps, capacity=sum(t))
    s = wl.spec
    o = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(s.batch, s.hq, dtype=torch.float32, device=DEV)
    ws = pkx.decode_attention_fwd(wl.q.to(DEV), o, kb.to(DEV), vb.to(DEV), kvp, kvi,
                                  wl.sm_scale, lse=lse)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    ko, vo = wl.pool()
    want_o, want_l = oracle.decode_attention(wl.q, ko, vo, wl.kv_indptr, wl.kv_indices,
                                             wl.sm_scale)
    assert_close(o.cpu(), lse.cpu(), want_o, want_l)


# ------------------------------------------------ KV write fused into extend
FUSED = [
    # (lq, lv, hq, hkv, prefix, extend) -- long prefixes make split-KV blocks
    (128, 128, 32, 8, [0, 1500, 300, 9000], [200, 64, 1, 130]),
    (64, 64, 12, 3, [999, 45, 0], [500, 2, 129]),
    (192, 128, 16, 4, [700, 33], [150, 64]),
    (288, 256, 16, 4, [129, 5], [70, 250]),
]


def _fused_case(wl, dev, fp8=None, scale=1.0):
    """Pool with the extend slots overwritten by stale rows; the fused call;
    returns (pool k, pool v, o, lse, ws) on the device and the oracle's
    expected pools."""
    k_ext, v_ext = wl.extend_kv()
    loc = wl.extend_kv_indices.to(torch.int64)
    if fp8 is None:
        kb, vb = wl.pool()
        kb = kb.clone()
        vb = vb if wl.spec.v_aliases_k else vb.clone()
        g = torch.Generator().manual_seed(3)
        kb[loc] = torch.randn(kb[loc].shape, generator=g).to(torch.bfloat16)
        if not wl.spec.v_aliases_k:
            vb[loc] = torch.randn(vb[loc].shape, generator=g).to(torch.bfloat16)
        else:
            vb = kb[..., : wl.spec.lv]
        want_k, want_v = oracle.set_kv_buffer(kb, vb, loc, k_ext,
                                              None if wl.spec.v_aliases_k else v_ext)
    else:
        kb, vb = wl.pool_fp8(fp8, scale, scale)
        kb.view(torch.uint8)[loc] = 0
        vb.view(torch.uint8)[loc] = 0
        want_k, want_v = oracle.set_kv_buffer_fp8(kb, vb, loc, k_ext, v_ext, scale, scale)
    dkb = kb.to(dev)
    dvb = dkb[..., : wl.spec.lv] if wl.spec.v_aliases_k else vb.to(dev)
    n = wl.n_q_tokens
    o = torch.full((n, wl.spec.hq, wl.spec.lv), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((n, wl.spec.hq), float("nan"), dtype=torch.float32, device=dev)
    kw = {} if fp8 is None else {"k_scale": scale, "v_scale": scale}
    dke = k_ext.to(dev)
    dve = dke[..., : wl.spec.lv] if wl.spec.v_aliases_k else v_ext.to(dev)
    ws = pkx.extend_attention_fwd(wl.q.to(dev), dke, dve, o, dkb, dvb,
                                  wl.qo_indptr.to(dev), wl.kv_indptr.to(dev),
                                  wl.kv_indices.to(dev), wl.sm_scale, wl.spec.logit_cap,
                                  wl.spec.sliding_window, lse=lse, cache_loc=loc.to(dev), **kw)
    torch.cuda.synchronize()
    return dkb, dvb, o, lse, ws, want_k, want_v


@pytest.mark.parametrize("lq,lv,hq,hkv,prefix,extend", FUSED)
def test_fused_kv_write_bit_exact_and_attention(lq, lv, hq, hkv, prefix, extend):
    """The two-stage call with cache_loc: the pool afterwards equals the
    oracle's set_kv_buffer bit for bit (every new row written once, nothing
    else touched), and o / lse match the oracle's two-stage attention."""
    from gpu_cases import assert_close, oracle_extend
    wl = W.draw(W.small_spec(batch=len(prefix), hq=hq, hkv=hkv, lq=lq, lv=lv, prefix=prefix,
                             extend=extend, seed=lq + sum(extend)))
    dkb, dvb, o, lse, ws, want_k, want_v = _fused_case(wl, DEV)
    assert pkx.workspace_status(ws) == 0
    assert torch.equal(dkb.cpu(), want_k)
    assert torch.equal(dvb.cpu(), want_v)
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, f"fused {lq}/{lv}")


def test_fused_kv_write_mla_and_fp8_fall_back_to_the_standalone_write():
    from gpu_cases import assert_close, oracle_extend
    spec = W.small_spec(batch=2, hq=16, hkv=1, lq=576, lv=512, prefix=[300, 20], extend=[40, 70],
                        std=0.5, v_aliases_k=True, sm_scale=1.0 / math.sqrt(192.0), seed=9)
    wl = W.draw(spec)
    dkb, dvb, o, lse, ws, want_k, _ = _fused_case(wl, DEV)
    assert pkx.workspace_status(ws) == 0
    assert torch.equal(dkb.cpu(), want_k)
    ro, rl = oracle_extend(wl)
    assert_close(o, lse, ro, rl, "fused mla")
    wl = W.draw(W.small_spec(batch=2, hq=8, hkv=2, lq=128, lv=128, prefix=[300, 20],
                             extend=[40, 70], seed=10))
    dkb, dvb, o, lse, ws, want_k, want_v = _fused_case(wl, DEV, fp8=torch.float8_e4m3fn,
                                                       scale=0.5)
    assert pkx.workspace_status(ws) == 0
    assert torch.equal(dkb.cpu().view(torch.uint8), want_k.view(torch.uint8))
    assert torch.equal(dvb.cpu().view(torch.uint8), want_v.view(torch.uint8))
    k_ext, v_ext = wl.extend_kv()
    ro, rl = oracle.extend_attention(wl.q, k_ext, v_ext, want_k, want_v, wl.qo_indptr,
                                     wl.kv_indptr, wl.kv_indices, wl.sm_scale, k_scale=0.5,
                                     v_scale=0.5)
    assert_close(o, lse, ro, rl, "fused fp8")


def test_fused_kv_write_full_size():
    """llama3_8b: the pool's extend slots are cleared, the fused call writes
    them back; the pool equals the workload's full pool bit for bit, and 2048
    sampled rows of o match the oracle."""
    from gpu_cases import assert_close, oracle_extend, sample_rows
    wl = W.draw(W.SPECS["llama3_8b"])
    kb, vb = wl.pool(DEV)
    full_k, full_v = kb.clone(), vb.clone()
    loc = wl.extend_kv_indices.to(torch.int64).to(DEV)
    kb[loc] = 0
    vb[loc] = 0
    k_ext, v_ext = wl.extend_kv(DEV)
    n = wl.n_q_tokens
    o = torch.empty(n, 32, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(n, 32, dtype=torch.float32, device=DEV)
    ws = pkx.extend_attention_fwd(wl.q.to(DEV), k_ext, v_ext, o, kb, vb, wl.qo_indptr.to(DEV),
                                  wl.kv_indptr.to(DEV), wl.kv_indices.to(DEV), wl.sm_scale,
                                  lse=lse, cache_loc=loc)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    assert torch.equal(kb, full_k) and torch.equal(vb, full_v)
    rows = sample_rows(n, 32, 2048, seed=82)
    ro, rl = oracle_extend(wl, rows=rows)
    assert_close(o.view(-1, 128)[rows.to(DEV)], lse.view(-1)[rows.to(DEV)], ro, rl, "fused full")
