"""The fp32 FMA throughput probe that prices the sparse FLOPs in the bench's
secondary step roofline: its outputs must be the chains it claims to run, so the
FLOP count it reports is work actually done. Each chain is replayed on the host in
float32 (fused multiply-add: exact float64 product plus addend, one rounding)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _fma32(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def _expected(n_threads, iters, chains=8):
    out = np.zeros(n_threads, dtype=np.float32)
    for tid in range(n_threads):
        seed = np.float32((tid & 1023) * 2.0 ** -12)
        m = np.float32(np.float32(0.5) + seed * np.float32(0.25))
        c = np.float32(np.float32(0.25) - seed)
        mul = (m, np.float32(m * np.float32(0.5)))
        add = (c, -c)
        s = np.float32(0.0)
        for k in range(chains):
            v = np.float32(seed + np.float32(k))
            lane = [v, -v]
            for _ in range(iters):
                lane = [_fma32(lane[0], mul[0], add[0]), _fma32(lane[1], mul[1], add[1])]
            s = np.float32(s + np.float32(lane[0] + lane[1]))
        out[tid] = s
    return out


def test_fma_probe_values_and_flops():
    blocks, iters = 2, 7
    out = torch.full((blocks * 256,), float("nan"), dtype=torch.float32, device="cuda")
    flops = tw.fma_probe(out, blocks, iters)
    torch.cuda.synchronize()
    assert flops == blocks * 256 * iters * 8 * 4
    np.testing.assert_allclose(out.cpu().numpy(), _expected(blocks * 256, iters), rtol=1e-6, atol=1e-6)


def test_fma_probe_rejects_bad_arguments():
    out = torch.empty(256, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        tw.fma_probe(out, 2, 1)          # out too small for 2 blocks
    with pytest.raises(tw.TwellError):
        tw.fma_probe(out, 1, 0)          # iters < 1


def test_l2_gather_probe_sums_the_gathered_rows():
    """Each thread's output is the sum of the eight bf16 columns it owns over every
    row index its CTA took, so the bytes it reports were gathered."""
    rng = np.random.default_rng(9)
    rows, d, n_idx, blocks = 300, 512, 8 * 37, 5
    tab = rng.integers(-8, 8, size=(rows, d)).astype(np.float32)   # small integers: every sum is exact
    bits = (tab.view(np.uint32) >> 16).astype(np.uint16)
    table = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    idx_np = rng.integers(0, rows, size=n_idx).astype(np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    out, nbytes = tw.l2_gather_probe(table, idx, blocks=blocks)
    torch.cuda.synchronize()
    assert nbytes == n_idx * d * 2
    exp = np.zeros((blocks, d // 8), dtype=np.float64)
    for g in range(n_idx // 8):
        b = g % blocks
        for r in idx_np[8 * g:8 * g + 8]:
            exp[b] += tab[r].reshape(d // 8, 8).sum(axis=1)
    np.testing.assert_array_equal(out.cpu().numpy().reshape(blocks, d // 8), exp.astype(np.float32))
