"""Seeded random sweeps of the helper kernels: pack / unpack of random
matrix sets (random owners, ranks, alignment, dtypes, matrices that start at
odd element offsets inside a larger allocation), and AdamW over random tensor
lists (odd sizes, unaligned views) against the fp64 oracle."""
import random

import numpy as np
import pytest

from oracle import adamw_oracle as ad
from oracle import muon_oracle as orc
from tests.gpu_util import to_f64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

INT = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32}


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


def _views(rng, g, shapes, dtype):
    """Matrices as views of one allocation, each at a random element offset."""
    offs, total = [], 0
    for s in shapes:
        total += rng.randint(0, 9)
        offs.append(total)
        total += s[0] * s[1]
    base = torch.randn(total + 16, generator=g, device="cuda").to(dtype)
    return [base[o:o + s[0] * s[1]].view(s) for o, s in zip(offs, shapes)]


@pytest.mark.parametrize("seed", range(6))
def test_random_pack(mg, seed):
    rng = random.Random(4400 + seed)
    g = torch.Generator(device="cuda").manual_seed(seed)
    dtype = rng.choice([torch.bfloat16, torch.float16, torch.float32])
    shapes = [(rng.randint(1, 900), rng.randint(1, 900)) for _ in range(rng.randint(1, 12))]
    ranks = rng.randint(1, 8)
    align = rng.choice([1, 8])
    owners = [rng.randrange(ranks) for _ in shapes]
    off, seg = mg.muon_pack_plan(shapes, owners, ranks, align)
    mats = _views(rng, g, shapes, dtype)
    sentinel = -777
    packed = torch.full((ranks * seg,), sentinel, dtype=INT[dtype], device="cuda").view(dtype)
    mg.muon_pack(mats, off, packed, to_packed=True)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    bits = packed.view(INT[dtype])
    covered = torch.zeros(ranks * seg, dtype=torch.bool, device="cuda")
    for i, t in enumerate(mats):
        n = t.numel()
        assert torch.equal(bits[off[i]:off[i] + n], t.reshape(-1).view(INT[dtype])), (seed, i)
        covered[off[i]:off[i] + n] = True
    assert bool((bits[~covered] == sentinel).all())
    back = _views(rng, g, shapes, dtype)
    mg.muon_pack(back, off, packed, to_packed=False)
    torch.cuda.synchronize()
    for a, b in zip(mats, back):
        assert torch.equal(a.view(INT[dtype]), b.view(INT[dtype]))


def _store(x64, dtype):
    return x64.astype(np.float32) if dtype == "f32" else orc.bf16_bits_from_f64(orc.round_bf16(x64))


@pytest.mark.parametrize("seed", range(6))
def test_random_adamw(mg, seed):
    rng = random.Random(5500 + seed)
    g = torch.Generator(device="cuda").manual_seed(100 + seed)
    pdt, sdt = rng.choice([("f32", "f32"), ("bf16", "f32"), ("bf16", "bf16")])
    tp = torch.float32 if pdt == "f32" else torch.bfloat16
    ts = torch.float32 if sdt == "f32" else torch.bfloat16
    sizes = [(1, rng.choice([1, 7, 33, 8192, 8193, rng.randint(1, 60000)])) for _ in range(rng.randint(1, 9))]
    p = [v.reshape(-1) for v in _views(rng, g, sizes, tp)]
    for v in p:
        v.mul_(0.5)
    m = [v.reshape(-1).zero_() for v in _views(rng, g, sizes, ts)]
    vv = [v.reshape(-1).zero_() for v in _views(rng, g, sizes, ts)]
    tol = 1e-5 if pdt == "f32" else 1e-3
    F = lambda x: float(np.float32(x))   # noqa: E731  hyper-parameters as the library receives them
    for t in (1, 2):
        lr, b1, b2, eps, wd = rng.choice([1e-3, 5e-4]), 0.9, rng.choice([0.99, 0.999]), 1e-8, rng.choice([0.0, 0.1])
        grads = [v.reshape(-1) * 0.1 for v in _views(rng, g, sizes, tp)]
        before = [(to_f64(a), to_f64(b), to_f64(c)) for a, b, c in zip(p, m, vv)]
        mg.muon_adamw_step(p, grads, m, vv, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=wd, step=t)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        for i in range(len(sizes)):
            p0, m0, v0 = before[i]
            gh = grads[i].cpu().float().numpy() if pdt == "f32" else \
                grads[i].cpu().view(torch.int16).numpy().view(np.uint16)
            ref = ad.adamw_step(_store(p0, pdt), gh, _store(m0, sdt), _store(v0, sdt),
                                lr=F(lr), beta1=F(b1), beta2=F(b2), eps=F(eps), wd=F(wd), step=t,
                                param_dtype=pdt, state_dtype=sdt)
            d = np.linalg.norm(ref["p_exact"] - ref["p_old"])
            if d == 0:
                continue
            err = np.linalg.norm(to_f64(p[i]) - ref["p_exact"]) / d
            q = np.linalg.norm(ref["p_new"] - ref["p_exact"]) / d
            assert err <= tol + q, (seed, t, i, sizes[i], err, q)
