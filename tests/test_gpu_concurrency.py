"""Host threads calling the library at the same time, each on its own stream
(the header allows that): every thread's Muon steps and NS calls must give
the same bytes as the same calls made one after another on one stream.  The
threads' shape mixes reach the product kernels, the fused small-matrix
kernel, the fp32 FFMA path and transposed layouts, so the per-stream
workspaces, tables and status word are all shared or raced for at once."""
import threading

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

STEPS = 3


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    yield pkg
    pkg.muon_set_ns_config(pkg.QUINTIC, 5, (2, 2, 1), pkg.MUON_PATH_AUTO)


# (shapes, parameter dtype, momentum dtype, NS input (batch, m, n)) per thread
JOBS = [
    ([(256, 1024), (1024, 256)], torch.bfloat16, torch.bfloat16, (2, 192, 640)),
    ([(128, 512)] * 6 + [(256, 256)] * 3, torch.bfloat16, torch.bfloat16, (4, 128, 512)),
    ([(768, 2048)], torch.bfloat16, torch.float32, (1, 512, 1536)),
    ([(300, 700), (700, 300), (37, 101)], torch.float32, torch.float32, (3, 96, 300)),
]


def _inputs(seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    out = []
    for shapes, pdt, mdt, xs in JOBS:
        W = [(torch.randn(s, generator=g, device="cuda") * 0.02).to(pdt) for s in shapes]
        M = [(torch.randn(s, generator=g, device="cuda") * 0.01).to(mdt) for s in shapes]
        G = [[(torch.randn(s, generator=g, device="cuda") * 0.03).to(pdt) for s in shapes] for _ in range(STEPS)]
        X = torch.randn(xs, generator=g, device="cuda").to(pdt)
        out.append((W, M, G, X))
    return out


def _work(mg, job, stream):
    W, M, G, X = job
    for t in range(STEPS):
        mg.muon_step(W, G[t], M, lr=0.02, beta=0.95, wd=0.1, nesterov=(t % 2 == 0), stream=stream)
    mg.muon_ns_orthogonalize(X, mg.QUINTIC, 5, (2, 2, 1), stream=stream)


def _clone(jobs):
    return [([w.clone() for w in W], [m.clone() for m in M], G, X.clone()) for W, M, G, X in jobs]


@pytest.mark.parametrize("path", ["plain", "gram"])
def test_threads_on_separate_streams_match_serial_calls(mg, path):
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM)
    base = _inputs(31 if path == "plain" else 32)
    serial = _clone(base)
    torch.cuda.synchronize()
    s0 = torch.cuda.Stream()
    for job in serial:
        _work(mg, job, s0)
    s0.synchronize()
    assert mg.muon_sync_status(s0) == mg.MUON_OK

    streams = [torch.cuda.Stream() for _ in base]
    # the first round starts on fresh streams (each grows its workspace while
    # the others compute), the second reuses them
    for rnd in range(2):
        jobs = _clone(base)
        torch.cuda.synchronize()
        start = threading.Barrier(len(jobs))
        errors = []

        def run(i):
            try:
                start.wait(timeout=60)
                with torch.cuda.stream(streams[i]):
                    _work(mg, jobs[i], streams[i])
                streams[i].synchronize()
            except Exception as e:        # noqa: BLE001 - reported on the main thread
                errors.append((i, repr(e)))

        threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
        for th in threads:
            th.start()
        for th in threads:
            th.join(timeout=300)
        assert not any(th.is_alive() for th in threads)
        assert not errors, errors
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        for i, ((W, M, _g, X), (Ws, Ms, _gs, Xs)) in enumerate(zip(jobs, serial)):
            for a, b in zip(W + M + [X], Ws + Ms + [Xs]):
                assert torch.equal(a, b), (path, rnd, i, tuple(a.shape), a.dtype)


def test_groups_in_threads_match_serial_steps(mg):
    """One persistent group per host thread (graph replay), stepped at the
    same time on separate streams, against muon_step made serially."""
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_GRAM)
    base = _inputs(33)
    serial = _clone(base)
    torch.cuda.synchronize()
    s0 = torch.cuda.Stream()
    for W, M, G, _x in serial:
        for t in range(STEPS):
            mg.muon_step(W, G[t], M, lr=0.01, beta=0.9, wd=0.05, nesterov=True, stream=s0)
    s0.synchronize()
    assert mg.muon_sync_status(s0) == mg.MUON_OK

    jobs = _clone(base)
    grads = [[g.clone() for g in G[0]] for _w, _m, G, _x in jobs]
    groups = [mg.MuonGroup(W, gr, M) for (W, M, _g, _x), gr in zip(jobs, grads)]
    streams = [torch.cuda.Stream() for _ in jobs]
    torch.cuda.synchronize()
    start = threading.Barrier(len(jobs))
    errors = []

    def run(i):
        try:
            start.wait(timeout=60)
            with torch.cuda.stream(streams[i]):
                for t in range(STEPS):
                    for dst, src in zip(grads[i], jobs[i][2][t]):
                        dst.copy_(src)          # the group reads its gradients in place
                    groups[i].step(lr=0.01, beta=0.9, wd=0.05, nesterov=True, stream=streams[i])
            streams[i].synchronize()
        except Exception as e:        # noqa: BLE001 - reported on the main thread
            errors.append((i, repr(e)))

    try:
        threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
        for th in threads:
            th.start()
        for th in threads:
            th.join(timeout=300)
        assert not any(th.is_alive() for th in threads)
        assert not errors, errors
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        for i, ((W, M, _g, _x), (Ws, Ms, _gs, _xs)) in enumerate(zip(jobs, serial)):
            for a, b in zip(W + M, Ws + Ms):
                assert torch.equal(a, b), (i, tuple(a.shape), a.dtype)
    finally:
        for grp in groups:
            grp.close()
