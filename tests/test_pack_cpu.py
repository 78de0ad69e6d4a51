"""The packed exchange layout (host-only, so it runs without a GPU): each
owner's matrices contiguous in its segment, segments of equal length, and a
two-rank gloo exchange over buffers in that layout hands every owner the sum
of its matrices' gradients (all-reduce, then each rank reads its segment:
what one reduce-scatter of the buffer delivers)."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402

SHAPES = [(2048, 2048), (1024, 4096), (7, 13), (4096, 1), (128, 512), (3, 3), (640, 200), (1, 9)]


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


@pytest.mark.parametrize("ranks,align", [(1, 8), (2, 8), (3, 1), (4, 32), (8, 8)])
def test_layout_invariants(mg, ranks, align):
    owners, _, _, _ = mg.muon_owner_plan(SHAPES, ranks)
    off, seg = mg.muon_pack_plan(SHAPES, owners, ranks, align)
    assert seg % align == 0
    sizes = [m * n for m, n in SHAPES]
    for r in range(ranks):
        mine = [i for i in range(len(SHAPES)) if owners[i] == r]
        # ascending index, aligned, inside the segment, disjoint and in order
        prev_end = r * seg
        for i in mine:
            assert (off[i] - r * seg) % align == 0
            assert off[i] >= prev_end and off[i] + sizes[i] <= (r + 1) * seg
            prev_end = off[i] + sizes[i]
    # the longest segment is tight: its last matrix ends within align of it
    longest = max((max((off[i] + sizes[i] - owners[i] * seg for i in range(len(SHAPES)) if owners[i] == r),
                       default=0)) for r in range(ranks))
    assert seg - longest < align
    # deterministic
    assert mg.muon_pack_plan(SHAPES, owners, ranks, align) == (off, seg)


def test_layout_rejects_bad_arguments(mg):
    with pytest.raises(mg.MuonError):
        mg.muon_pack_plan([(4, 4)], [2], 2)          # owner out of range
    with pytest.raises(mg.MuonError):
        mg.muon_pack_plan([(0, 4)], [0], 1)          # zero side
    with pytest.raises(mg.MuonError):
        mg.muon_pack_plan([(4, 4)], [0], 0)          # no ranks
    with pytest.raises(mg.MuonError):
        mg.muon_pack_plan([(4, 4)], [0], 1, 0)       # alignment
    assert mg.muon_pack_plan([], [], 3) == ([], 0)


def test_pack_rejects_overflowing_sizes(mg):
    """Sizes whose byte range overflows int64 are rejected before any device
    use.  The matrix and buffer pointers are placeholders, so this runs only
    where no CUDA device is present: a validation bug then fails with a
    missing-device status instead of reaching a kernel."""
    import ctypes
    if torch.cuda.is_available():
        pytest.skip("placeholder pointers: host-only check")
    L = mg.lib()
    fake = ctypes.c_void_p(4096)
    big = (1 << 62)
    for m, n, off in ((big, 4, 0), (1 << 31, 1 << 31, 0), (4, 4, (1 << 63) - 8), (1 << 30, 1 << 27, 0)):
        r = L.muon_pack((ctypes.c_void_p * 1)(fake), (ctypes.c_int64 * 1)(m), (ctypes.c_int64 * 1)(n),
                        (ctypes.c_int64 * 1)(off), 1, mg.MUON_BF16, fake, 1, None)
        assert r == mg.MUON_EINVAL, (m, n, off, r)
        assert "overflow" in mg.last_error_message() or "too many" in mg.last_error_message()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import newton_schulz_frobenius_gb300 as mg
    shapes = SHAPES[2:]                       # small enough for CPU buffers
    owners, _, _, _ = mg.muon_owner_plan(shapes, world)
    off, seg = mg.muon_pack_plan(shapes, owners, world, 8)
    # this rank's gradients (a rank-dependent seed), packed by the layout
    g = torch.Generator().manual_seed(100 + rank)
    grads = [torch.randn(m * n, generator=g, dtype=torch.float64) for m, n in shapes]
    buf = torch.zeros(world * seg, dtype=torch.float64)
    for i, t in enumerate(grads):
        buf[off[i]:off[i] + t.numel()] = t
    dist.all_reduce(buf)
    mine = buf[rank * seg:(rank + 1) * seg].clone()
    out[rank] = (owners, off, seg, mine.numpy().tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_exchange_over_the_layout():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    shapes = SHAPES[2:]
    owners, off, seg, _ = out[0]
    assert out[1][:3] == (owners, off, seg)       # both ranks computed the same layout
    # regenerate each rank's gradients and sum them per matrix
    per_rank = []
    for r in range(2):
        g = torch.Generator().manual_seed(100 + r)
        per_rank.append([torch.randn(m * n, generator=g, dtype=torch.float64) for m, n in shapes])
    for r in range(2):
        mine = np.array(out[r][3])
        for i in range(len(shapes)):
            if owners[i] != r:
                continue
            lo = off[i] - r * seg
            np.testing.assert_array_equal(mine[lo:lo + shapes[i][0] * shapes[i][1]],
                                          (per_rank[0][i] + per_rank[1][i]).numpy())


@pytest.mark.parametrize("ranks,align", [(1, 1), (2, 8), (3, 4), (8, 32)])
def test_layout_matches_oracle(mg, ranks, align):
    """The library's planner against the oracle's plain restatement of the
    layout, on owners from the owner planner and on a skewed hand-made
    assignment (every matrix on the last rank but one)."""
    from oracle import pack_oracle as po
    owners, _, _, _ = mg.muon_owner_plan(SHAPES, ranks)
    assert mg.muon_pack_plan(SHAPES, owners, ranks, align) == tuple(po.layout(SHAPES, owners, ranks, align))
    skew = [ranks - 1] * len(SHAPES)
    skew[0] = 0
    assert mg.muon_pack_plan(SHAPES, skew, ranks, align) == tuple(po.layout(SHAPES, skew, ranks, align))


def test_oracle_pack_places_every_element():
    from oracle import pack_oracle as po
    shapes, owners = [(2, 3), (1, 5), (3, 1)], [1, 0, 1]
    off, seg = po.layout(shapes, owners, 2, 4)
    # rank 0: matrix 1 at 0, ends at 5 (8 with alignment); rank 1: matrix 0 at 0,
    # ends at 6, matrix 2 at 8, ends at 11 (12): segments of 12
    assert (off, seg) == ([12, 0, 20], 12)
    mats = [np.arange(m * n, dtype=np.float64).reshape(m, n) + 10 * i for i, (m, n) in enumerate(shapes)]
    buf = po.pack(mats, off, 2 * seg, fill=-1)
    for a, o in zip(mats, off):
        np.testing.assert_array_equal(buf[o:o + a.size], a.reshape(-1))
    assert (buf == -1).sum() == 2 * seg - sum(a.size for a in mats)


def _owner_step_worker(rank, world, port, out):
    """One owner-centric Muon step over CPU ranks: gradients summed into the
    packed layout, each owner updating its matrices (the fp64 oracle stands in
    for the per-owner GPU update), updated parameters published through the
    same layout."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import newton_schulz_frobenius_gb300 as mg
    from oracle import muon_oracle as orc
    shapes = [(16, 48), (40, 24), (8, 8), (24, 72)]
    owners, _, _, _ = mg.muon_owner_plan(shapes, world, mg.MUON_F32)
    off, seg = mg.muon_pack_plan(shapes, owners, world, 4)
    W = [np.random.default_rng(7 + i).standard_normal(s).astype(np.float32) * 0.02 for i, s in enumerate(shapes)]
    G = [np.random.default_rng(100 * rank + i).standard_normal(s).astype(np.float32) * 0.01
         for i, s in enumerate(shapes)]
    # 1. gradients summed into their owners' segments (one reduction of the buffer)
    gbuf = torch.zeros(world * seg, dtype=torch.float32)
    for i, g in enumerate(G):
        gbuf[off[i]:off[i] + g.size] = torch.from_numpy(g.reshape(-1))
    dist.all_reduce(gbuf)
    # 2. each owner updates its matrices; 3. published through the same layout
    pbuf = torch.zeros(world * seg, dtype=torch.float32)
    for i, (m, n) in enumerate(shapes):
        if owners[i] != rank:
            continue
        gsum = gbuf[off[i]:off[i] + m * n].numpy().reshape(m, n)
        r = orc.muon_step(W[i], np.zeros((m, n), np.float32), gsum, lr=0.02, beta=0.95, wd=0.1, nesterov=False,
                          path="gram" if m != n else "plain", param_dtype="f32", mom_dtype="f32")
        pbuf[off[i]:off[i] + m * n] = torch.from_numpy(np.asarray(r["W_new"], np.float32).reshape(-1))
    dist.all_reduce(pbuf)                     # every segment filled by its owner alone
    out[rank] = [pbuf[off[i]:off[i] + m * n].numpy().reshape(m, n).tolist() for i, (m, n) in enumerate(shapes)]
    dist.barrier()
    dist.destroy_process_group()


def test_owner_centric_step_over_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    world = 2
    mp.start_processes(_owner_step_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    from oracle import muon_oracle as orc
    shapes = [(16, 48), (40, 24), (8, 8), (24, 72)]
    for i, (m, n) in enumerate(shapes):
        a, b = np.array(out[0][i]), np.array(out[1][i])
        np.testing.assert_array_equal(a, b)             # every rank holds the same parameters
        W = np.random.default_rng(7 + i).standard_normal((m, n)).astype(np.float32) * 0.02
        gsum = sum(np.random.default_rng(100 * r + i).standard_normal((m, n)).astype(np.float32) * 0.01
                   for r in range(world)).astype(np.float32)
        ref = orc.muon_step(W, np.zeros((m, n), np.float32), gsum, lr=0.02, beta=0.95, wd=0.1, nesterov=False,
                            path="gram" if m != n else "plain", param_dtype="f32", mom_dtype="f32")
        np.testing.assert_array_equal(a, np.asarray(ref["W_new"], np.float32))
