"""Persistent groups (muon_group_*): a registered set of matrices stepped many
times must give exactly the results of muon_step on the same inputs, with the
hyper-parameters changing from step to step, whether the steps replay a
captured CUDA graph or launch directly."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    yield pkg
    pkg.muon_set_ns_config(pkg.QUINTIC, 5, (2, 2, 1), pkg.MUON_PATH_AUTO)


def _make(shapes, pdt, mdt, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    W = [(torch.randn(s, generator=g, device="cuda") * 0.02).to(pdt) for s in shapes]
    G = [(torch.randn(s, generator=g, device="cuda") * 0.03).to(pdt) for s in shapes]
    M = [torch.zeros(s, device="cuda", dtype=mdt) for s in shapes]
    return W, G, M


SHAPES = [(128, 512), (512, 128), (128, 512), (256, 640), (640, 256), (96, 96), (1, 24)]
SCHEDULE = [(0.02, 0.95, 0.1, True), (0.01, 0.9, 0.05, False), (0.03, 0.95, 0.0, True), (0.015, 0.8, 0.1, True)]


@pytest.mark.parametrize("graph", ["1", "0"])
@pytest.mark.parametrize("mdt", [torch.bfloat16, torch.float32])
def test_group_matches_muon_step(mg, monkeypatch, graph, mdt):
    monkeypatch.setenv("MUON_GRAPH", graph)
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_AUTO)
    Wa, Ga, Ma = _make(SHAPES, torch.bfloat16, mdt, 11)
    Wb, Gb, Mb = [w.clone() for w in Wa], [g.clone() for g in Ga], [m.clone() for m in Ma]
    group = mg.MuonGroup(Wb, Gb, Mb)
    try:
        for i, (lr, beta, wd, nest) in enumerate(SCHEDULE):
            # fresh gradients each step, written in place
            for ga, gb in zip(Ga, Gb):
                ga.mul_(-0.7).add_(0.001 * (i + 1))
                gb.copy_(ga)
            mg.muon_step(Wa, Ga, Ma, lr=lr, beta=beta, wd=wd, nesterov=nest)
            group.step(lr=lr, beta=beta, wd=wd, nesterov=nest)
            torch.cuda.synchronize()
            assert mg.muon_sync_status() == mg.MUON_OK
            for x, y in zip(Wa + Ma, Wb + Mb):
                assert torch.equal(x, y), i
    finally:
        group.close()


def test_group_counts_its_launches_and_replans(mg, monkeypatch):
    monkeypatch.setenv("MUON_GRAPH", "1")
    W, G, M = _make([(256, 640), (128, 512)], torch.bfloat16, torch.bfloat16, 5)
    group = mg.MuonGroup(W, G, M)
    try:
        group.step(lr=0.02)                       # direct
        c0 = mg.muon_launch_count()
        group.step(lr=0.02)                       # captures and replays
        c1 = mg.muon_launch_count()
        group.step(lr=0.01)                       # replays
        c2 = mg.muon_launch_count()
        assert c1 - c0 == c2 - c1 > 0
        mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_PLAIN)   # plans change
        group.step(lr=0.01)
        assert mg.muon_last_path(256, 640, mg.MUON_BF16) == mg.MUON_PATH_PLAIN
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
    finally:
        group.close()
        mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_AUTO)


def test_group_validation(mg):
    W, G, M = _make([(64, 64)], torch.bfloat16, torch.bfloat16, 3)
    with pytest.raises(ValueError):
        mg.MuonGroup([], [], [])
    with pytest.raises(mg.MuonError):
        h = mg.MuonGroup(W, G, M)
        mg.muon_group_step(h.handle, float("nan"), 0.9, 0.0, False)


def test_group_fused_buckets_match_step(mg, monkeypatch):
    """Five fused buckets of both forms (128-row and 256-row) in one fused
    launch with work lists, replayed from the group's graph: bitwise the same
    weights and momenta as muon_step on the same inputs."""
    monkeypatch.setenv("MUON_SMALL", "1")
    monkeypatch.setenv("MUON_GRAPH", "1")
    shapes = [(128, 512)] * 5 + [(256, 256)] * 3 + [(192, 256), (512, 128), (256, 200), (64, 96)]
    W1, G1, M1 = _make(shapes, torch.bfloat16, torch.bfloat16, 31)
    W2, G2, M2 = [w.clone() for w in W1], [g.clone() for g in G1], [m.clone() for m in M1]
    group = mg.MuonGroup(W1, G1, M1)
    try:
        for _ in range(3):
            group.step(lr=0.02, beta=0.95, wd=0.1, nesterov=False)
            mg.muon_step(W2, G2, M2, lr=0.02, beta=0.95, wd=0.1, nesterov=False)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        for a, b in zip(W1 + M1, W2 + M2):
            assert torch.equal(a, b)
    finally:
        group.close()


@pytest.mark.parametrize("graph", ["1", "0"])
def test_group_host_io_overlapped(mg, monkeypatch, graph):
    """Host-resident gradients and parameters (muon_group_set_host_io): every
    step copies the gradients in from pinned host memory and the updated
    parameters out, chunk by chunk on the group's copy streams.  Over several
    steps with gradients rewritten on the host, the device weights and momenta
    equal those of muon_step on device gradients, and the host parameters
    equal the device weights after every step."""
    monkeypatch.setenv("MUON_GRAPH", graph)
    monkeypatch.setenv("MUON_WORKSPACE_MB", "2")      # several chunks per bucket
    shapes = [(256, 640), (640, 256), (256, 640), (128, 512), (512, 128), (96, 96)] * 2
    Wa, Ga, Ma = _make(shapes, torch.bfloat16, torch.float32, 71)
    Wb, Mb = [w.clone() for w in Wa], [m.clone() for m in Ma]
    Gb = [torch.zeros_like(g) for g in Ga]             # filled from the host every step
    host_g = [g.cpu().pin_memory() for g in Ga]
    host_w = [torch.empty_like(w, device="cpu").pin_memory() for w in Wb]
    group = mg.MuonGroup(Wb, Gb, Mb)
    try:
        group.set_host_io(host_g, host_w)
        for i, (lr, beta, wd, nest) in enumerate(SCHEDULE):
            for ga, hg in zip(Ga, host_g):
                ga.mul_(-0.7).add_(0.001 * (i + 1))
                hg.copy_(ga)                          # the host holds this step's gradients
            torch.cuda.synchronize()
            mg.muon_step(Wa, Ga, Ma, lr=lr, beta=beta, wd=wd, nesterov=nest)
            group.step(lr=lr, beta=beta, wd=wd, nesterov=nest)
            torch.cuda.synchronize()
            assert mg.muon_sync_status() == mg.MUON_OK
            for x, y in zip(Wa + Ma, Wb + Mb):
                assert torch.equal(x, y), i
            for hw, w in zip(host_w, Wb):
                assert torch.equal(hw, w.cpu()), i
        # copies off again: the group steps on its device gradients
        group.set_host_io(None, None)
        group.step(lr=0.02)
        mg.muon_step(Wa, Gb, Ma, lr=0.02, beta=0.95, wd=0.0, nesterov=True)
        torch.cuda.synchronize()
        for x, y in zip(Wa + Ma, Wb + Mb):
            assert torch.equal(x, y)
    finally:
        group.close()


def test_group_host_io_rejects_pageable_memory(mg):
    W, G, M = _make([(64, 128)], torch.bfloat16, torch.bfloat16, 9)
    group = mg.MuonGroup(W, G, M)
    try:
        with pytest.raises(mg.MuonError) as ei:
            group.set_host_io([G[0].cpu()], None)        # pageable
        assert ei.value.status == mg.MUON_EINVAL
        with pytest.raises(ValueError):
            group.set_host_io([G[0].cpu().pin_memory()] * 2, None)
    finally:
        group.close()
