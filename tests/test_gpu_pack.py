"""The pack kernel on the GPU: matrices into a packed buffer laid out by
muon_pack_plan and back, bit for bit, the padding between them untouched;
16-byte and element paths, every storage type, matrices of several chunks."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SHAPES = [(300, 700), (7, 13), (4096, 1), (128, 512), (3, 3), (640, 200), (1, 9), (2048, 40)]
INT = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32}


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_pack_round_trip(mg, dtype, align):
    owners, _, _, _ = mg.muon_owner_plan(SHAPES, 3)
    off, seg = mg.muon_pack_plan(SHAPES, owners, 3, align)
    g = torch.Generator(device="cuda").manual_seed(5)
    mats = [torch.randn(s, generator=g, device="cuda").to(dtype) for s in SHAPES]
    sentinel = -12345
    packed = torch.full((3 * seg,), sentinel, dtype=INT[dtype], device="cuda").view(dtype)
    mg.muon_pack(mats, off, packed, to_packed=True)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    bits = packed.view(INT[dtype])
    covered = torch.zeros(3 * seg, dtype=torch.bool, device="cuda")
    for i, t in enumerate(mats):
        n = t.numel()
        assert torch.equal(bits[off[i]:off[i] + n], t.reshape(-1).view(INT[dtype]))
        covered[off[i]:off[i] + n] = True
    assert bool((bits[~covered] == sentinel).all())          # padding untouched
    back = [torch.zeros_like(t) for t in mats]
    mg.muon_pack(back, off, packed, to_packed=False)
    torch.cuda.synchronize()
    for a, b in zip(mats, back):
        assert torch.equal(a.view(INT[dtype]), b.view(INT[dtype]))


def test_pack_rejects_mismatch(mg):
    a = torch.zeros((4, 4), device="cuda", dtype=torch.bfloat16)
    buf = torch.zeros(8, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mg.muon_pack([a], [0], buf)                           # does not fit
    with pytest.raises(TypeError):
        mg.muon_pack([a], [0], torch.zeros(64, device="cuda", dtype=torch.float32))
