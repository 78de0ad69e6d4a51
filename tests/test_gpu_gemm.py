"""Kernel-level tests of the product kernels through muon_debug_gemm, against a
plain PyTorch reference of the same product (fp64 on the GPU from the same
stored operands).  bf16 runs on the tcgen05 tensor-core kernel, fp32 on the
FFMA kernel.  Shapes span several tiles and ragged tails."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * scale).to(dtype)


def _check(C, ref, dtype):
    C64 = C.double()
    err = (C64 - ref).norm() / ref.norm()
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-5
    assert err.item() < tol, err.item()
    # elementwise: within a few output ulps of the reference scale
    scale = ref.abs().max().item()
    atol = (2.0 ** -6 if dtype == torch.bfloat16 else 1e-5) * scale
    assert (C64 - ref).abs().max().item() <= atol


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K,batch,tile", [
    (128, 128, 64, 1, 0), (256, 512, 320, 2, 256), (256, 512, 320, 2, 128),
    (200, 264, 136, 3, 0), (384, 1000, 72, 1, 128), (1, 8, 8, 1, 0)])
def test_product_k_major(mg, dtype, M, N, K, batch, tile):
    A = _rand((batch, M, K), dtype, 1)
    B = _rand((batch, N, K), dtype, 2)
    C = torch.zeros((batch, M, N), dtype=dtype, device="cuda")
    mg.muon_debug_gemm(A, B, C, b_kmajor=True, alpha=0.5, tile_n=tile)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    ref = 0.5 * torch.matmul(A.double(), B.double().transpose(1, 2))
    _check(C, ref, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K,batch,tile", [
    (128, 256, 128, 1, 256), (200, 304, 136, 2, 256), (200, 304, 136, 2, 128),
    (512, 1000, 512, 1, 0), (64, 64, 64, 1, 128)])
def test_product_mn_major(mg, dtype, M, N, K, batch, tile):
    A = _rand((batch, M, K), dtype, 3)
    B = _rand((batch, K, N), dtype, 4)
    C = torch.zeros((batch, M, N), dtype=dtype, device="cuda")
    mg.muon_debug_gemm(A, B, C, b_kmajor=False, tile_n=tile)
    torch.cuda.synchronize()
    ref = torch.matmul(A.double(), B.double())
    _check(C, ref, dtype)


@pytest.mark.parametrize("kmajor", [True, False])
@pytest.mark.parametrize("M,N,K,batch", [(64, 64, 1000, 1), (128, 192, 520, 1), (100, 70, 776, 2), (256, 1024, 256, 1),
                                          (72, 90, 1001, 1)])
def test_fp32_split_k(mg, kmajor, M, N, K, batch):
    """fp32 products with few output tiles split K over clusters of CTAs
    (ragged k-ranges, 16-byte and scalar loads); the partial tiles are added
    in a fixed order, so two runs agree bit for bit."""
    A = _rand((batch, M, K), torch.float32, 21)
    B = _rand((batch, N, K) if kmajor else (batch, K, N), torch.float32, 22)
    C = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    mg.muon_debug_gemm(A, B, C, b_kmajor=kmajor)
    C2 = torch.zeros_like(C)
    mg.muon_debug_gemm(A, B, C2, b_kmajor=kmajor)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    assert torch.equal(C, C2)
    Bd = B.double().transpose(1, 2) if kmajor else B.double()
    _check(C, torch.matmul(A.double(), Bd), torch.float32)


@pytest.mark.parametrize("kmajor", [True, False])
@pytest.mark.parametrize("M,N,K,batch", [(1536, 1664, 200, 1), (1500, 1701, 77, 1), (700, 900, 130, 4)])
def test_fp32_large_tiles(mg, kmajor, M, N, K, batch):
    """fp32 products with at least one 128 x 128 tile per SM run on the
    large-tile FFMA kernel: ragged edges, odd K and pitches, batches."""
    A = _rand((batch, M, K), torch.float32, 31)
    B = _rand((batch, N, K) if kmajor else (batch, K, N), torch.float32, 32)
    C = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    mg.muon_debug_gemm(A, B, C, b_kmajor=kmajor, alpha=0.5)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    Bd = B.double().transpose(1, 2) if kmajor else B.double()
    _check(C, 0.5 * torch.matmul(A.double(), Bd), torch.float32)


def test_fp32_large_tiles_symmetric(mg):
    X = _rand((1, 2304, 136), torch.float32, 33)
    C = torch.full((1, 2304, 2304), float("nan"), dtype=torch.float32, device="cuda")
    mg.muon_debug_gemm(X, X, C, b_kmajor=True, symmetric=True)
    torch.cuda.synchronize()
    assert torch.equal(C, C.transpose(1, 2))
    _check(C, torch.matmul(X.double(), X.double().transpose(1, 2)), torch.float32)


def test_fp32_split_k_symmetric(mg):
    X = _rand((1, 96, 1000), torch.float32, 23)
    C = torch.full((1, 96, 96), float("nan"), dtype=torch.float32, device="cuda")
    mg.muon_debug_gemm(X, X, C, b_kmajor=True, symmetric=True)
    torch.cuda.synchronize()
    assert torch.equal(C, C.transpose(1, 2))
    _check(C, torch.matmul(X.double(), X.double().transpose(1, 2)), torch.float32)


@pytest.mark.parametrize("tile", [128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("m,k,batch", [(128, 64, 1), (260, 1000, 2), (512, 384, 1), (37, 200, 3), (896, 136, 1)])
def test_symmetric_gram(mg, dtype, m, k, batch, tile):
    """Lower-triangle tiles of 128 x 128 or 128 x 256, mirrored on store."""
    if dtype == torch.bfloat16 and k % 8:
        pytest.skip("tensor-map rows need 16-byte pitch")
    X = _rand((batch, m, k), dtype, 5)
    C = torch.full((batch, m, m), float("nan"), dtype=dtype, device="cuda")
    mg.muon_debug_gemm(X, X, C, b_kmajor=True, symmetric=True, alpha=1.0 / k, tile_n=tile)
    torch.cuda.synchronize()
    assert torch.equal(C, C.transpose(1, 2))          # mirrored, every element written
    ref = torch.matmul(X.double(), X.double().transpose(1, 2)) / k
    _check(C, ref, dtype)


@pytest.mark.parametrize("tile", [128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("m", [128, 384, 200])
def test_fused_polynomial(mg, dtype, m, tile):
    X = _rand((1, m, 2 * m), torch.float64, 6)
    G64 = torch.matmul(X, X.transpose(1, 2))
    G64 = G64 / torch.linalg.matrix_norm(G64, ord=2, keepdim=True)
    G = G64.to(dtype).contiguous()
    P = torch.zeros_like(G)
    a, b, c = 3.4445, -4.7750, 2.0315
    mg.muon_debug_gemm(G, G, P, b_kmajor=True, symmetric=True, poly=(a, b, c), tile_n=tile)
    torch.cuda.synchronize()
    Gd = G.double()
    ref = a * torch.eye(m, device="cuda", dtype=torch.float64) + b * Gd + c * torch.matmul(Gd, Gd)
    assert torch.equal(P, P.transpose(1, 2))
    _check(P, ref, dtype)


def test_large_gram_and_apply_bf16(mg):
    """The two long products at the 2560 x 9728 size (several waves of tiles)."""
    m, n = 2560, 9728
    X = _rand((1, m, n), torch.bfloat16, 7, scale=1.0 / np.sqrt(n))
    G = torch.zeros((1, m, m), dtype=torch.bfloat16, device="cuda")
    mg.muon_debug_gemm(X, X, G, b_kmajor=True, symmetric=True)
    Q = _rand((1, m, m), torch.bfloat16, 8, scale=1.0 / np.sqrt(m))
    Y = torch.zeros((1, m, n), dtype=torch.bfloat16, device="cuda")
    mg.muon_debug_gemm(Q, X, Y, b_kmajor=False)
    torch.cuda.synchronize()
    Xd = X.double()
    _check(G, torch.matmul(Xd, Xd.transpose(1, 2)), torch.bfloat16)
    _check(Y, torch.matmul(Q.double(), Xd), torch.bfloat16)


def _tf32_rne(t):
    u = t.view(torch.int32)
    u = (u + 0xFFF + ((u >> 13) & 1)) & ~0x1FFF
    return u.view(torch.float32)


def _tf32_trunc(t):
    """fp32 values with the 13 low mantissa bits cleared (the TF32 operand)."""
    return (t.view(torch.int32) & ~0x1FFF).view(torch.float32)


@pytest.mark.parametrize("M,N,K,batch,sym", [
    (128, 128, 32, 1, False), (256, 384, 200, 2, False), (200, 200, 200, 1, True), (384, 384, 520, 2, True)])
def test_product_tf32(mg, M, N, K, batch, sym):
    A = _rand((batch, M, K), torch.float32, 9)
    B = A if sym else _rand((batch, N, K), torch.float32, 10)
    C = torch.zeros((batch, M, N), dtype=torch.float32, device="cuda")
    mg.muon_debug_gemm(A, B, C, b_kmajor=True, symmetric=sym, tf32=True)
    torch.cuda.synchronize()
    exact = torch.matmul(A.double(), B.double().transpose(1, 2))
    err = ((C.double() - exact).norm() / exact.norm()).item()
    assert err < 2e-3, err                      # TF32 operands: 10-bit mantissa
    if sym:
        assert torch.equal(C, C.transpose(1, 2))
    # the product of the TF32 operands (low mantissa bits dropped or rounded
    # off, whichever the hardware does) accumulated in fp32 matches closely
    errs = []
    for conv in (_tf32_trunc, _tf32_rne):
        At, Bt = conv(A.contiguous()).double(), conv(B.contiguous()).double()
        near = torch.matmul(At, Bt.transpose(1, 2))
        errs.append(((C.double() - near).norm() / near.norm()).item())
    assert min(errs) < 1e-5, errs


def test_poly_tf32(mg):
    m = 256
    X = _rand((1, m, 3 * m), torch.float64, 11)
    G = torch.matmul(X, X.transpose(1, 2))
    G = (G / torch.linalg.matrix_norm(G, ord=2, keepdim=True)).float().contiguous()
    P = torch.zeros_like(G)
    a, b, c = 3.4445, -4.7750, 2.0315
    mg.muon_debug_gemm(G, G, P, b_kmajor=True, symmetric=True, poly=(a, b, c), tf32=True)
    torch.cuda.synchronize()
    Gd = G.double()
    ref = a * torch.eye(m, device="cuda", dtype=torch.float64) + b * Gd + c * torch.matmul(Gd, Gd)
    err = ((P.double() - ref).norm() / ref.norm()).item()
    assert err < 2e-3, err


@pytest.mark.parametrize("kind,M,N,K,batch", [
    ("kmajor", 256, 512, 320, 2), ("kmajor", 384, 1000, 136, 1), ("kmajor", 200, 264, 72, 3),
    ("sym", 896, 896, 136, 1), ("sym", 384, 384, 1000, 2), ("sym", 260, 260, 200, 1),
    ("mn", 200, 304, 136, 2), ("mn", 640, 1000, 512, 1), ("mn", 384, 256, 256, 3),
    ("tf32", 384, 384, 520, 2), ("tf32sym", 896, 896, 136, 1)])
def test_paired_products(mg, monkeypatch, kind, M, N, K, batch):
    """128 x 256 tiles run as 2-SM products on 2-CTA clusters (row blocks 2p
    and 2p+1; each CTA loads its own A rows and its half of the B tile; an odd
    last block reads zeros and stores nothing), and, with MUON_MC=1, as 4-CTA
    clusters of two pairs on tiles that share their A rows, each A row loaded
    once per cluster by TMA multicast (an odd tile count leaves one pair
    repeating its partner's tile without storing it).  Same tiles and K order
    as the unpaired kernel, so all three results are bitwise equal, and they
    match the fp64 product."""
    tf32 = kind.startswith("tf32")
    dtype = torch.float32 if tf32 else torch.bfloat16
    sym = kind in ("sym", "tf32sym")
    kmajor = kind != "mn"
    A = _rand((batch, M, K), dtype, 21, scale=1.0 / np.sqrt(K))
    B = A if sym else (_rand((batch, N, K), dtype, 22) if kmajor else _rand((batch, K, N), dtype, 23))
    out = []
    for pair, mc in (("0", "0"), ("1", "0"), ("1", "1")):
        monkeypatch.setenv("MUON_PAIR", pair)
        monkeypatch.setenv("MUON_MC", mc)
        C = torch.full((batch, M, N), float("nan"), dtype=dtype, device="cuda")
        mg.muon_debug_gemm(A, B, C, b_kmajor=kmajor, symmetric=sym, tile_n=256, tf32=tf32)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        out.append(C)
    assert torch.equal(out[0], out[1])
    assert torch.equal(out[0], out[2])
    Bt = B.double().transpose(1, 2) if kmajor else B.double()
    ref = torch.matmul(A.double(), Bt)
    if tf32:
        err = ((out[1].double() - ref).norm() / ref.norm()).item()
        assert err < 2e-3, err
    else:
        _check(out[1], ref, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind,M,N,K,batch,tile", [
    ("sym", 264, 264, 200, 2, 256), ("sym", 896, 896, 136, 1, 128), ("sym", 384, 384, 520, 1, 256),
    ("kmajor", 200, 264, 136, 3, 256), ("kmajor", 384, 1000, 72, 1, 128), ("poly", 296, 296, 0, 2, 256)])
def test_tile_store_epilogue(mg, monkeypatch, dtype, kind, M, N, K, batch, tile):
    """16-bit workspace products leave the kernel as 32 x 32 tile stores (a chunk
    below the diagonal also as its transpose, the diagonal chunk assembled
    symmetric).  They write the same values as the staged row stores
    (MUON_TMA_STORE=0), bit for bit, cover every element of a ragged output
    (C starts as NaN) and keep a symmetric product exactly symmetric."""
    poly = kind == "poly"
    sym = kind in ("sym", "poly")
    if poly:
        X = _rand((batch, M, 2 * M), torch.float64, 41)
        G = torch.matmul(X, X.transpose(1, 2))
        A = (G / torch.linalg.matrix_norm(G, ord=2, keepdim=True)).to(dtype).contiguous()
        B = A
    else:
        A = _rand((batch, M, K), dtype, 42, scale=1.0 / np.sqrt(K))
        B = A if sym else _rand((batch, N, K), dtype, 43)
    out = []
    for flag in ("0", "1"):
        monkeypatch.setenv("MUON_TMA_STORE", flag)
        C = torch.full((batch, M, N), float("nan"), dtype=dtype, device="cuda")
        if poly:
            mg.muon_debug_gemm(A, B, C, b_kmajor=True, symmetric=True, poly=(3.4445, -4.7750, 2.0315), tile_n=tile)
        else:
            mg.muon_debug_gemm(A, B, C, b_kmajor=True, symmetric=sym, tile_n=tile)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        out.append(C)
    assert not torch.isnan(out[1]).any()
    assert torch.equal(out[0], out[1])
    if sym:
        assert torch.equal(out[1], out[1].transpose(1, 2))
    Ad = A.double()
    if poly:
        a, b, c = 3.4445, -4.7750, 2.0315
        ref = a * torch.eye(M, device="cuda", dtype=torch.float64) + b * Ad + c * torch.matmul(Ad, Ad)
    else:
        ref = torch.matmul(Ad, B.double().transpose(1, 2))
    err = ((out[1].double() - ref).norm() / ref.norm()).item()
    assert err < (1e-2 if dtype == torch.bfloat16 else 2e-3), err
