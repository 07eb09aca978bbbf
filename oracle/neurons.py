"""Per-neuron activity counts and dead-neuron re-initialisation of the gate
projection (test infrastructure only; see the package docstring).

The pages report that aggressive L1 leaves "dead" neurons that never fire, and that
targeted re-initialisation of the gate projection's weights mitigates them
(thelatestinai listing, Table 5 "Dead neuron reinit." row and caption, Figure 8;
wispaper blog "Critical Analysis & Conclusion"; gist.science explainer, "Future
Directions"). They do not give the re-initialisation distribution or the window over
which a neuron counts as dead. This build's reading: a neuron is dead for a step when
no token activates it (a_tj = ReLU(g_tj) > 0 for no t); its gate row Wg[j, :] is
redrawn as std * z with z from a fixed, reproducible generator: the Irwin-Hall sum of
twelve uniforms minus 6 (mean 0, variance 1, support [-6, 6]), the uniforms taken
from SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the constants of its reference implementation) used as a
counter-based generator. Every step of that is exact integer or float64
arithmetic, so the CUDA kernel's values must match bit for bit.
"""
from __future__ import annotations

import numpy as np

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def splitmix64_at(seed: int, counter: np.ndarray) -> np.ndarray:
    """The counter-th output (0-based) of a SplitMix64 generator seeded with `seed`:
    state = seed + (counter + 1) * gamma (mod 2^64), then the output mix."""
    c = np.asarray(counter, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK) + (c + np.uint64(1)) * np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def reinit_values(seed: int, rows: np.ndarray, d: int, std: float) -> np.ndarray:
    """bf16 bit patterns of the re-drawn rows [len(rows), d]: element (j, k) uses
    counters 12 (j d + k) + i, i < 12; u_i = (top 24 bits) / 2^24;
    z = sum u_i - 6 (exact in float64); w = float32(float64(std) * z), then bf16
    round to nearest even."""
    rows = np.asarray(rows, dtype=np.uint64)
    k = np.arange(d, dtype=np.uint64)
    base = (rows[:, None] * np.uint64(d) + k[None, :]) * np.uint64(12)
    total = np.zeros(base.shape, dtype=np.int64)
    for i in range(12):
        total += (splitmix64_at(seed, base + np.uint64(i)) >> np.uint64(40)).astype(np.int64)
    z = total.astype(np.float64) / float(1 << 24) - 6.0
    w = (np.float64(np.float32(std)) * z).astype(np.float32)
    bits = w.view(np.uint32).astype(np.uint64)
    # round to nearest even on the upper 16 bits (finite values only here)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    return ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def neuron_counts(a: np.ndarray) -> np.ndarray:
    """counts[j] = number of tokens t with a[t, j] > 0 (a dense activation matrix as
    float values or bf16 bit patterns; for bits, nonzero magnitude bits)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return ((a & 0x7FFF) != 0).sum(axis=0).astype(np.int64)
    return (a > 0).sum(axis=0).astype(np.int64)


def reinit_dead_rows(W: np.ndarray, counts: np.ndarray, seed: int, std: float) -> tuple[np.ndarray, int]:
    """W (bf16 bits [I, d]) with every row j of counts[j] == 0 redrawn; returns the new
    matrix and the number of rows redrawn."""
    W = np.array(W, dtype=np.uint16, copy=True)
    dead = np.flatnonzero(np.asarray(counts) == 0)
    if dead.size:
        W[dead] = reinit_values(seed, dead, W.shape[1], std)
    return W, int(dead.size)
