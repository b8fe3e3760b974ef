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


def test_no_alloc_decode_matches_workspace_decode_twice():
    dev = torch.device("cuda:0")
    wl, kb, vb, q, kvp, kvi = _decode_inputs(dev)
    s = wl.spec
    o_ref = torch.empty(s.batch, s.hq, s.lv, dtype=torch.bfloat16, device=dev)
    l_ref = torch.empty(s.batch, s.hq, dtype=torch.float32, device=dev)
    pkx.decode_attention_fwd(q, o_ref, kb, vb, kvp, kvi, wl.sm_scale, s.logit_cap, lse=l_ref)
    for _ in range(2):  # two calls in a row share (and reuse) the scratch
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(l_ref, float("nan"))
        pkx.decode_attention_fwd_no_alloc(q, o, kb, vb, kvp, kvi, wl.sm_scale, s.logit_cap, lse=lse)
        torch.cuda.synchronize()
        err = (o.float() - o_ref.float()).abs()
        assert torch.isfinite(o.float()).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
        assert (lse - l_ref).abs().max().item() <= LSE_ABS


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
