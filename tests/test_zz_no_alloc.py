"""The allocation-free decode entry point (pkx_decode_attention_fwd_no_alloc).

Callers that cannot allocate device memory (a plugin whose host framework
owns all device memory, a decode loop that must not call cudaMalloc because
it synchronises the device) use this variant; its scratch is a fixed array
inside the library.  This file is named so that pytest collects it last.
"""
import pytest
import torch

from paged_kv_extend_gb300 import pkx
from paged_kv_extend_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkx.load_library()


def _decode_inputs(dev):
    spec = W.WorkloadSpec("dec", batch=12, hq=32, hkv=8, lq=128, lv=128,
                          prefix=[0, 5, 130, 4095, 777, 2048, 1, 9000, 63, 64, 300, 1500],
                          extend=[1] * 12, num_slots=1 << 16, logit_cap=30.0, seed=99,
                          decode=True)
    wl = W.draw(spec)
    kb, vb = wl.pool(dev)
    return wl, kb, vb, wl.q.to(dev), wl.kv_indptr.to(dev), wl.kv_indices.to(dev)


def _assert_close(o, lse, ref_o, ref_lse):
    o, lse = o.double().cpu(), lse.double().cpu()
    ref_o, ref_lse = ref_o.double().cpu(), ref_lse.double().cpu()
    err = (o - ref_o).abs()
    assert torch.isfinite(o).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse - ref_lse).abs().max().item() <= LSE_ABS


def test_no_alloc_decode_matches_workspace_decode_twice():
    """Two calls in a row (sharing and reusing the scratch) against the
    workspace call and against the float64 oracle; the status word of the
    built-in scratch reads clean after each."""
    import oracle
    dev = torch.device("cuda:0")
    wl, kb, vb, q, kvp, kvi = _decode_inputs(dev)
    s = wl.spec
    o_ref = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
    l_ref = torch.empty(s.batch, s.hq, dtype=torch.float32, device=dev)
    pkx.decode_attention_fwd(q, o_ref, kb, vb, kvp, kvi, wl.sm_scale, s.logit_cap, lse=l_ref)
    ckb, cvb = wl.pool()
    ro, rl = oracle.decode_attention(wl.q, ckb, cvb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     s.logit_cap)
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(l_ref, float("nan"))
        pkx.decode_attention_fwd_no_alloc(q, o, kb, vb, kvp, kvi, wl.sm_scale, s.logit_cap, lse=lse)
        torch.cuda.synchronize()
        assert pkx.decode_no_alloc_status() == pkx.PKX_OK
        _assert_close(o, lse, o_ref, l_ref)
        _assert_close(o, lse, ro, rl)


def test_no_alloc_reports_device_status():
    """An index outside the pool is not read; the call records PKX_EDEVICE in
    the built-in scratch's status word, which decode_no_alloc_status reads
    back, and the next good call clears it."""
    dev = torch.device("cuda:0")
    wl, kb, vb, q, kvp, kvi = _decode_inputs(dev)
    s = wl.spec
    bad = kvi.clone()
    bad[5] = kb.shape[0] + 77
    o = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
    pkx.decode_attention_fwd_no_alloc(q, o, kb, vb, kvp, bad, wl.sm_scale, s.logit_cap)
    assert pkx.decode_no_alloc_status() == pkx.PKX_EDEVICE
    assert torch.isfinite(o.float()).all()
    pkx.decode_attention_fwd_no_alloc(q, o, kb, vb, kvp, kvi, wl.sm_scale, s.logit_cap)
    assert pkx.decode_no_alloc_status() == pkx.PKX_OK


def test_no_alloc_rejects_problem_beyond_scratch():
    """A problem whose scratch exceeds the built-in array is refused before
    anything runs (real, valid tensors: no sequence has any key)."""
    dev = torch.device("cuda:0")
    h, d = 128, 128
    batch = 1000
    while pkx.decode_workspace_min_size(batch, h, h, d, d) <= (96 << 20):
        batch *= 2
        assert batch <= (1 << 17)
    q = torch.zeros(batch, h, d, dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    kb = torch.zeros(8, h, d, dtype=torch.bfloat16, device=dev)
    kvp = torch.zeros(batch + 1, dtype=torch.int32, device=dev)
    kvi = torch.zeros(0, dtype=torch.int32, device=dev)
    with pytest.raises(pkx.PkxError) as e:
        pkx.decode_attention_fwd_no_alloc(q, o, kb, kb, kvp, kvi)
    assert e.value.code == pkx.PKX_EWORKSPACE
    assert "scratch" in str(e.value)


def test_no_alloc_falls_back_to_one_key_stream():
    """A batch whose two-stream scratch exceeds the built-in array but whose
    one-stream scratch fits runs with one key stream per unit, and matches
    the workspace call (two streams)."""
    dev = torch.device("cuda:0")
    hq, hkv, d, t = 32, 8, 128, 40
    batch = 256
    while pkx.decode_workspace_size(batch, hq, hkv, d, d) <= (96 << 20):
        batch *= 2
    assert pkx.decode_workspace_min_size(batch, hq, hkv, d, d) <= (96 << 20)
    g = torch.Generator().manual_seed(5)
    slots = batch * t
    kb = torch.randn(slots, hkv, d, generator=g).to(torch.bfloat16).to(dev)
    vb = torch.randn(slots, hkv, d, generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn(batch, hq, d, generator=g).to(torch.bfloat16).to(dev)
    lens = torch.randint(1, t + 1, (batch,), generator=g)
    kvp = torch.cat([torch.zeros(1, dtype=torch.int64), lens.cumsum(0)]).to(torch.int32).to(dev)
    kvi = torch.randperm(slots, generator=g)[: int(lens.sum())].to(torch.int32).to(dev)
    o_ref = torch.empty(batch, hq, d, dtype=torch.bfloat16, device=dev)
    l_ref = torch.empty(batch, hq, dtype=torch.float32, device=dev)
    pkx.decode_attention_fwd(q, o_ref, kb, vb, kvp, kvi, lse=l_ref)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(l_ref, float("nan"))
    pkx.decode_attention_fwd_no_alloc(q, o, kb, vb, kvp, kvi, lse=lse)
    torch.cuda.synchronize()
    err = (o.float() - o_ref.float()).abs()
    assert torch.isfinite(o.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse - l_ref).abs().max().item() <= LSE_ABS


@pytest.mark.parametrize("dt", [torch.float8_e4m3fn, torch.float8_e5m2])
def test_fp8_decode_with_one_stream_workspace(dt):
    """Decode over an fp8 pool given only decode_workspace_min_size bytes: one
    key stream per unit, whose products run in f16 like the two-stream path
    (the codes' values, the query times 2^-8), against the oracle."""
    import oracle
    dev = torch.device("cuda:0")
    lens = [1, 130, 2049, 700]
    hq, hkv, d, ks, vs = 16, 2, 128, 0.1, 0.04
    spec = W.WorkloadSpec("dec", batch=len(lens), hq=hq, hkv=hkv, lq=d, lv=d,
                          prefix=[t - 1 for t in lens], extend=[1] * len(lens),
                          num_slots=2 * sum(lens) + 16, logit_cap=30.0, seed=71, decode=True)
    wl = W.draw(spec)
    kb, vb = wl.pool_fp8(dt, ks, vs)
    ro, rl = oracle.decode_attention(wl.q, kb, vb, wl.kv_indptr, wl.kv_indices, wl.sm_scale,
                                     30.0, -1, k_scale=ks, v_scale=vs)
    n_min = pkx.decode_workspace_min_size(wl.batch, hq, hkv, d, d)
    assert n_min < pkx.decode_workspace_size(wl.batch, hq, hkv, d, d)
    ws = torch.empty(n_min, dtype=torch.uint8, device=dev)
    o = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    pkx.decode_attention_fwd(wl.q.to(dev), o, kb.to(dev), vb.to(dev), wl.kv_indptr.to(dev),
                             wl.kv_indices.to(dev), wl.sm_scale, 30.0, lse=lse, workspace=ws,
                             k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws) == 0
    err = (o.float().cpu() - ro.float()).abs()
    assert torch.isfinite(o.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (lse.cpu() - rl.float()).abs().max().item() <= LSE_ABS
