"""Owner placement (muon_owner_plan) on the CPU: no GPU, no tune cache, so the
per-matrix costs are the algorithmic FLOPs of the path the library would pick
(Gram 2+2+1 when n > m, plain otherwise), checked here against the oracle's own
product log.  The plan is the greedy longest-processing-time-first fallback of
the pages' owner placement ("DMuon" news page, section 3; summary, section 2.3)."""
import itertools
import os
import socket

import pytest

from oracle import muon_oracle as orc
from workloads import WORKLOADS


@pytest.fixture(scope="module")
def mg():
    from newton_schulz_frobenius_gb300 import _build
    _build.build()
    import newton_schulz_frobenius_gb300 as pkg
    pkg.lib()
    return pkg


def _oracle_cost(r, c):
    m, n = min(r, c), max(r, c)
    path = "gram" if n > m else "plain"
    return orc.ns_product_log(m, n, path).algorithmic_flops()


SMALL = [(64, 256), (128, 128), (96, 300), (32, 512), (200, 200), (48, 64), (128, 512), (80, 80)]


def test_loads_are_the_oracle_costs(mg):
    owners, loads, mk, measured = mg.muon_owner_plan(SMALL, 3)
    assert not measured
    want = [0.0] * 3
    for (r, c), o in zip(SMALL, owners):
        want[o] += _oracle_cost(r, c)
    assert all(abs(a - b) <= 1e-9 * b for a, b in zip(loads, want))
    assert mk == max(loads)


def test_greedy_rule(mg):
    owners, _, _, _ = mg.muon_owner_plan(SMALL, 3)
    costs = [_oracle_cost(r, c) for r, c in SMALL]
    order = sorted(range(len(SMALL)), key=lambda i: -costs[i])    # stable: ties keep index order
    load = [0.0] * 3
    for i in order:
        best = min(range(3), key=lambda k: (load[k], k))
        assert owners[i] == best
        load[best] += costs[i]


@pytest.mark.parametrize("ranks", [2, 3])
def test_within_graham_bound_of_optimum(mg, ranks):
    shapes = SMALL[:7]
    costs = [_oracle_cost(r, c) for r, c in shapes]
    opt = min(max(sum(c for c, o in zip(costs, assign) if o == k) for k in range(ranks))
              for assign in itertools.product(range(ranks), repeat=len(costs)))
    _, _, mk, _ = mg.muon_owner_plan(shapes, ranks)
    assert opt <= mk <= (4.0 / 3.0 - 1.0 / (3 * ranks)) * opt + 1e-6 * opt


def test_seven_b_stack_beats_round_robin(mg):
    wl = WORKLOADS["stack_32L_7b_bf16_f32mom"]
    shapes = [(r, c) for _, r, c in wl.matrices()]
    costs = [_oracle_cost(r, c) for r, c in shapes]
    owners, loads, mk, _ = mg.muon_owner_plan(shapes, 8)
    rr = [0.0] * 8
    for i, c in enumerate(costs):
        rr[i % 8] += c
    assert mk <= max(rr)
    lower = max(sum(costs) / 8, max(costs))
    assert mk <= 4.0 / 3.0 * lower
    assert sorted(set(owners)) == list(range(8))


def test_degenerate_inputs(mg):
    owners, loads, mk, _ = mg.muon_owner_plan([], 4)
    assert owners == [] and loads == [0.0] * 4 and mk == 0.0
    owners, _, _, _ = mg.muon_owner_plan([(10, 10)], 5)
    assert owners == [0]
    with pytest.raises(mg.MuonError):
        mg.muon_owner_plan([(10, 10)], 0)
    with pytest.raises(mg.MuonError):
        mg.muon_owner_plan([(10, (1 << 20) + 1)], 2)      # beyond the library's side limit
    owners, _, _, _ = mg.muon_owner_plan([(1 << 20, 1 << 20)], 2)
    assert owners == [0]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from newton_schulz_frobenius_gb300 import _build
    _build.build()
    import newton_schulz_frobenius_gb300 as pkg
    wl = WORKLOADS["stack_24L_h2048_bf16"]
    shapes = [(r, c) for _, r, c in wl.matrices()]
    owners, _, _, _ = pkg.muon_owner_plan(shapes, world)
    mine = [i for i, o in enumerate(owners) if o == rank]
    gathered = [None] * world
    dist.all_gather_object(gathered, (owners, mine))
    out[rank] = gathered
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_owners(mg):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    g0, g1 = out[0], out[1]
    assert g0 == g1
    (owners_a, mine_a), (owners_b, mine_b) = g0
    assert owners_a == owners_b                                   # same plan on every rank
    assert sorted(mine_a + mine_b) == list(range(len(owners_a)))  # a partition of the matrices
