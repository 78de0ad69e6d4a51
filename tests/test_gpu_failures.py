"""Failure paths reported as status codes, with no GPU fault: every device
allocation of the library's own storage fails (MUON_FAIL_ALLOC=1, the
allocator hook), and the calls that need new storage return MUON_ENOMEM
without launching anything; once allocation works again, the same calls on
the same stream succeed."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


def _mats(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn(shape, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    gr = (torch.randn(shape, generator=g, device="cuda") * 0.03).to(torch.bfloat16)
    return w, gr, torch.zeros_like(w)


def test_workspace_allocation_failure(mg, monkeypatch):
    stream = torch.cuda.Stream()            # a stream with no workspace yet
    w, g, m = _mats((256, 1024), 1)
    w0 = w.clone()
    monkeypatch.setenv("MUON_FAIL_ALLOC", "1")
    before = mg.muon_launch_count()
    with pytest.raises(mg.MuonError) as ei:
        mg.muon_step([w], [g], [m], lr=0.02, beta=0.95, wd=0.1, nesterov=False, stream=stream)
    assert ei.value.status == mg.MUON_ENOMEM
    assert mg.muon_launch_count() == before
    torch.cuda.synchronize()
    assert torch.equal(w, w0)                # nothing was written
    monkeypatch.delenv("MUON_FAIL_ALLOC")
    mg.muon_step([w], [g], [m], lr=0.02, beta=0.95, wd=0.1, nesterov=False, stream=stream)
    stream.synchronize()
    assert mg.muon_sync_status(stream) == mg.MUON_OK
    assert not torch.equal(w, w0)


def test_group_allocation_failure(mg, monkeypatch):
    w, g, m = _mats((384, 768), 2)
    monkeypatch.setenv("MUON_FAIL_ALLOC", "1")
    with pytest.raises(mg.MuonError) as ei:
        grp = mg.MuonGroup([w], [g], [m])
        grp.step(lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert ei.value.status == mg.MUON_ENOMEM
    monkeypatch.delenv("MUON_FAIL_ALLOC")
    grp = mg.MuonGroup([w], [g], [m])
    try:
        grp.step(lr=0.02, beta=0.95, wd=0.1, nesterov=False)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
    finally:
        grp.close()
