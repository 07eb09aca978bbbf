"""GPU parity of the per-neuron activity counts and of the dead-neuron
re-initialisation against oracle/neurons.py. The counts kernel is fed a seeded
synthetic Hybrid (random ELL rows and dense backup rows built on the host, no FFN
arithmetic), so its expected counts are exact; after a real forward, the counts must
add up to the Hybrid's stored entries."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import activation_sparse_feedforward_gb300 as tw  # noqa: E402
from gpu_util import bits_of, to_dev  # noqa: E402
from oracle import neurons  # noqa: E402
from synthetic import FFNSpec, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    tw.load()


def _synthetic_hybrid(T, I, R, cap, n_backup, seed):
    """A Hybrid filled on the host: ELL rows with random distinct ascending neurons,
    backup rows with random fp32 a of which about 30% are > 0, and the dense matrix
    of nonzero activations it encodes."""
    rng = np.random.default_rng(seed)
    h = tw.Hybrid.empty(T, I, R, cap, gated=True, device="cuda")
    dense = np.zeros((T, I), dtype=bool)
    backup_rows = np.sort(rng.choice(T, n_backup, replace=False))
    ell_nnz = np.zeros(T, dtype=np.int32)
    ell_idx = np.zeros((T, R), dtype=np.uint16)
    slot = np.full(T, -1, dtype=np.int32)
    for t in range(T):
        if t in backup_rows:
            continue
        n = int(rng.integers(0, R + 1))
        cols = np.sort(rng.choice(I, n, replace=False))
        ell_nnz[t] = n
        ell_idx[t, :n] = cols
        dense[t, cols] = True
    ba = rng.standard_normal((max(cap, 1), I)).astype(np.float32) - 0.5
    for s, t in enumerate(backup_rows):
        slot[t] = s
        dense[t] = ba[s] > 0
    h.ell_nnz.copy_(torch.from_numpy(ell_nnz))
    h.ell_idx.copy_(torch.from_numpy(ell_idx.view(np.int16)))
    h.backup_slot.copy_(torch.from_numpy(slot))
    h.backup_a.copy_(torch.from_numpy(ba))
    h.n_backup.fill_(n_backup)
    return h, dense


@pytest.mark.parametrize("T,I,R,cap,nb", [(300, 704, 24, 16, 9), (1000, 5632, 64, 8, 0), (257, 1280, 100, 40, 40)])
def test_counts_match_oracle_on_a_synthetic_hybrid(T, I, R, cap, nb):
    h, dense = _synthetic_hybrid(T, I, R, cap, nb, seed=T + I)
    counts = torch.full((I,), 5, dtype=torch.int32, device="cuda")     # accumulates onto what is there
    tw.hybrid_neuron_counts(h, counts)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(counts.cpu().numpy(), neurons.neuron_counts(dense) + 5)


def test_counts_after_a_forward_add_up_to_the_stored_entries():
    spec = FFNSpec("counts_fwd", T=777, d=512, I=1280, mean_active=20, outlier_frac=0.03, W=128, C=8, R=48, seed=5)
    inp = make_inputs(spec)
    hf = tw.HybridFFN(spec.T, spec.d, spec.I, spec.W, spec.C, spec.R, spec.T // 4)
    hf.forward(*(to_dev(inp[k]) for k in ("x", "Wg", "Wu", "Wd")))
    counts = tw.hybrid_neuron_counts(hf.saved)
    torch.cuda.synchronize()
    tw.raise_if_device_error(hf.status)
    s = hf.saved
    nb = int(s.n_backup.item())
    stored = int(s.ell_nnz.sum().item()) + int((s.backup_a[:nb] > 0).sum().item())
    assert int(counts.sum().item()) == stored and nb > 0


@pytest.mark.parametrize("I,d,seed,std", [(700, 256, 1, 0.02), (64, 2048, 0xDEADBEEFCAFEF00D, 1.0)])
def test_reinit_matches_oracle_bit_for_bit(I, d, seed, std):
    rng = np.random.default_rng(I)
    W = rng.integers(0, 1 << 16, size=(I, d), dtype=np.uint16)
    counts = (rng.integers(0, 4, size=I) * (rng.random(I) < 0.6)).astype(np.int32)
    Wd = to_dev(W)
    n = tw.reinit_dead_rows(Wd, torch.from_numpy(counts).cuda(), seed, std)
    torch.cuda.synchronize()
    ref, n_ref = neurons.reinit_dead_rows(W, counts, seed, std)
    assert int(n.item()) == n_ref > 0
    np.testing.assert_array_equal(bits_of(Wd), ref)
