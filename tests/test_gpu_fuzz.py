"""Seeded random sweep of the product kernels through muon_debug_gemm:
shapes, batches, operand layouts, tile widths, symmetric and polynomial
products, bf16 / fp16 on the tensor-core kernel (and TF32 for fp32 operands),
fp32 on the FFMA kernel, against the same product in fp64 from the stored
operands.  Every draw respects the documented operand rules (16-byte rows on
the tensor-core path, K-major B for TF32), so each call must succeed."""
import random

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = {"bf16": 1e-2, "f16": 4e-3, "f32": 1e-5, "tf32": 3e-3}


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


def _draw(rng):
    kind = rng.choice(["bf16", "f16", "f32", "tf32"])
    sym = rng.random() < 0.35
    poly = sym and rng.random() < 0.4
    align = {"bf16": 8, "f16": 8, "f32": 1, "tf32": 4}[kind]
    M = rng.randint(1, 520)
    K = max(align, rng.randint(1, 1100) // align * align)
    if poly:
        K = M = max(align, M // align * align)
    N = M if sym else rng.randint(1, 700)
    kmajor = True if (sym or kind == "tf32") else rng.random() < 0.5
    if not kmajor:
        N = max(align, N // align * align)
    batch = rng.choice([1, 1, 2, 3])
    tile = rng.choice([0, 128, 256])
    return kind, M, N, K, batch, sym, poly, kmajor, tile


@pytest.mark.parametrize("seed", range(6))
def test_random_products(mg, seed):
    rng = random.Random(1000 + seed)
    g = torch.Generator(device="cuda").manual_seed(seed)
    for _ in range(8):
        kind, M, N, K, batch, sym, poly, kmajor, tile = _draw(rng)
        dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32, "tf32": torch.float32}[kind]
        A = (torch.randn((batch, M, K), generator=g, device="cuda") / K ** 0.5).to(dt)
        if poly:
            A = ((A.double() + A.double().transpose(1, 2)) * 0.5).to(dt).contiguous()
        B = A if sym else (torch.randn((batch, N, K) if kmajor else (batch, K, N), generator=g, device="cuda")
                           / K ** 0.5).to(dt)
        C = torch.full((batch, M, N), float("nan"), dtype=dt, device="cuda")
        coeffs = (3.4445, -4.7750, 2.0315) if poly else None
        mg.muon_debug_gemm(A, B, C, b_kmajor=kmajor, symmetric=sym, poly=coeffs, tile_n=tile,
                           tf32=(kind == "tf32"))
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        Ad = A.double()
        Bd = B.double().transpose(1, 2) if kmajor else B.double()
        ref = torch.matmul(Ad, Bd)
        if poly:
            a, b, c = coeffs
            ref = a * torch.eye(M, device="cuda", dtype=torch.float64) + b * Ad + c * ref
        case = (kind, M, N, K, batch, sym, poly, kmajor, tile)
        assert not torch.isnan(C).any(), case
        if sym:
            assert torch.equal(C, C.transpose(1, 2)), case
        err = ((C.double() - ref).norm() / ref.norm().clamp_min(1e-30)).item()
        assert err < TOL[kind], (case, err)


@pytest.mark.parametrize("seed", range(4))
def test_random_fp32_large_products(mg, seed):
    """fp32 products with at least one 128x128 tile per SM (the large-tile
    FFMA kernel): ragged M, N and K, both B layouts, symmetric and
    polynomial products, one or two matrices."""
    rng = random.Random(2000 + seed)
    g = torch.Generator(device="cuda").manual_seed(50 + seed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for _ in range(3):
        sym = rng.random() < 0.4
        poly = sym and rng.random() < 0.5
        batch = rng.choice([1, 2])
        M = rng.randint(1700, 2400) if not sym else rng.randint(2050, 2500)
        K = M if poly else rng.randint(1, 600)
        N = M if sym else rng.randint(1700, 2400)
        kmajor = True if sym else rng.random() < 0.5
        bm, bn = -(-M // 128), -(-N // 128)
        assert (bm * (bm + 1) // 2 if sym else bm * bn) * batch >= sms
        A = torch.randn((batch, M, K), generator=g, device="cuda") / K ** 0.5
        if poly:
            A = ((A + A.transpose(1, 2)) * 0.5).contiguous()
        B = A if sym else torch.randn((batch, N, K) if kmajor else (batch, K, N), generator=g,
                                      device="cuda") / K ** 0.5
        C = torch.full((batch, M, N), float("nan"), device="cuda")
        coeffs = (3.4445, -4.7750, 2.0315) if poly else None
        mg.muon_debug_gemm(A, B, C, b_kmajor=kmajor, symmetric=sym, poly=coeffs)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        Ad = A.double()
        ref = torch.matmul(Ad, B.double().transpose(1, 2) if kmajor else B.double())
        if poly:
            a, b, c = coeffs
            ref = a * torch.eye(M, device="cuda", dtype=torch.float64) + b * Ad + c * ref
        case = (M, N, K, batch, sym, poly, kmajor)
        assert not torch.isnan(C).any(), case
        if sym:
            assert torch.equal(C, C.transpose(1, 2)), case
        err = ((C.double() - ref).norm() / ref.norm()).item()
        assert err < TOL["f32"], (case, err)
