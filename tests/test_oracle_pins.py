"""The fp64 oracle against its pins (CPU only)."""
import math

import numpy as np
import pytest

from oracle import bruteforce
from tests import _pins
from tests._golden import load_cases


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin):
    pin(oracle_mod)


def test_bruteforce_golden():
    """The brute force itself reproduces the hand-worked cases."""
    for c in load_cases():
        d = c["d"]
        if c["kind"] == "full":
            z, _ = bruteforce.read([list(s) for s in c["src"]], list(c["w"][0]), list(c["gamma"]), c["eps"])
            assert np.max(np.abs(np.array(z) - c["expect"][0])) <= c["tol"], c["name"]
        else:
            N, S = c["N"], c["S"]
            W = [list(c["w_all"])] * (N * S)
            G = [list(c["gamma"])] * (N * S)
            out = bruteforce.block_pass(list(c["src"][0]), [list(s) for s in c["src"][1:]], S, W, G, c["eps"])
            assert np.max(np.abs(np.array(out) - c["expect"])) <= c["tol"], c["name"]


def _count_sources(orc, monkeypatch, fn):
    counts = []
    real = orc.read

    def counting(sources, *a, **k):
        counts.append(len(sources))
        return real(sources, *a, **k)

    monkeypatch.setattr(orc, "read", counting)
    fn()
    return counts


@pytest.mark.parametrize("L", [2, 4, 8, 32])
def test_source_counts_match_flop_accounting(oracle_mod, monkeypatch, L):
    """Source counts reproduce the pages' FLOP accounting (DepthBench reading
    notes section 4.7, paper Appendix D).

    Full: Delta F_Full = 4 T d L (2L + 3) counts 4d flops per (read, source) over
    the 2L sublayer reads and the LM-head read, leaving out the first sublayer,
    which reads the embedding alone (an identity). Block: Delta F_Block =
    4 T d [sum_{k=1}^{2L-1} (2 + floor(k/b)) + 9], b = 2L/8, counts the running
    sum at every sublayer; under the reading that an empty running sum is no
    source, the counts are that total minus the 7 interior block starts.
    """
    d, T = 2, 1
    R = 2 * L + 1
    hist = np.ones((R, T, d))
    W = np.zeros((R, d))
    G = np.ones((R, d))
    full_counts = _count_sources(oracle_mod, monkeypatch,
                                 lambda: oracle_mod.full_pass(hist, R, W, G, 1e-6))
    assert full_counts == list(range(1, R + 1))
    assert sum(c for c in full_counts if c >= 2) == L * (2 * L + 3)

    if (2 * L) % 8 == 0:
        b = 2 * L // 8
        monkeypatch.undo()
        emb = np.ones((T, d))
        F = np.ones((2 * L, T, d))
        blk_counts = _count_sources(
            oracle_mod, monkeypatch,
            lambda: oracle_mod.block_pass(emb, F, 8, b, W[: 2 * L], G[: 2 * L], 1e-6))
        head = 1 + 8
        pages = sum(2 + k // b for k in range(1, 2 * L)) + 9
        ours = sum(blk_counts[1:]) + head
        assert pages - ours == 7


def test_parameter_overhead_matches_table6():
    """Per-read w and gamma: 2 (2L + 1) d parameters. At the 24-layer shape
    (d = 1024) that is 0.10M, the Full/Block AttnRes delta over Pre-LN in the
    DepthBench reading notes, section 5 (paper Table 6: 405.41M -> 405.51M)."""
    L, d = 24, 1024
    extra = 2 * (2 * L + 1) * d
    assert round(extra / 1e6, 2) == round(405.51 - 405.41, 2)


def test_oracle_rejects_bad_arguments(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.read([], np.zeros(2), np.ones(2), 1e-6)
    with pytest.raises(ValueError):
        oracle_mod.read([np.zeros((2, 3))], np.zeros(3), np.ones(3), 1e-6, rows=[5])
    with pytest.raises(ValueError):
        oracle_mod.read([np.zeros((2, 3)), np.zeros((2, 4))], np.zeros(3), np.ones(3), 1e-6)


def test_oracle_threads(oracle_mod):
    assert oracle_mod.threads() >= 1
