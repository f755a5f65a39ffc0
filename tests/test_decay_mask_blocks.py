"""The block decomposition of the 128 x 128 decay mask that the tensor-core
sweep's P step uses, checked on the CPU against the mask's definition
(gamma^(p(i) - p(j)) where p(j) <= p(i), else 0).  Rows i = 32 q + lane and keys
j = 32 b + jj fall in 32 x 32 blocks, each of them one of:
  zero      keys on the masked side of the diagonal block row;
  diagonal  gamma^|lane - jj| on the unmasked side, 0 on the other;
  rank one  forward gamma^(32(q - b) + lane - 31) * gamma^(31 - jj),
            reverse gamma^(32(b - q) - lane) * gamma^jj;
with every factor a non-negative power of gamma, so none exceeds 1.  A chunk
shorter than 128 tokens uses the same blocks, then clears rows past its end
(forward) or keys past it (reverse)."""
import numpy as np
import pytest


def block_mask(gamma, reverse, Lc=128):
    M = np.zeros((128, 128))
    worst_exponent = np.inf
    for q in range(4):
        for b in range(4):
            for lane in range(32):
                for jj in range(32):
                    i, j = 32 * q + lane, 32 * b + jj
                    if q == b:
                        ok = jj >= lane if reverse else jj <= lane
                        M[i, j] = gamma ** abs(lane - jj) if ok else 0.0
                    elif (b > q) == reverse:
                        e1, e2 = ((32 * (b - q) - lane, jj) if reverse else
                                  (32 * (q - b) + lane - 31, 31 - jj))
                        worst_exponent = min(worst_exponent, e1, e2)
                        M[i, j] = gamma ** e1 * gamma ** e2
    if reverse:
        M[:, Lc:] = 0.0
    else:
        M[Lc:, :] = 0.0
    return M, worst_exponent


def reference_mask(gamma, reverse, Lc=128):
    # token positions 0..127 of the chunk; a reversed chunk processes its tokens
    # last to first, so p = Lc - 1 - position, and positions >= Lc are absent
    pos = np.arange(128)
    p = (Lc - 1 - pos) if reverse else pos
    valid = pos < Lc
    m = p[:, None] - p[None, :]
    keep = (m >= 0) & valid[:, None] & valid[None, :]
    return np.where(keep, gamma ** np.maximum(m, 0), 0.0)


@pytest.mark.parametrize("gamma", [1.0, 0.97, 0.5, np.exp(-6.56)])
@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("Lc", [128, 77, 1])
def test_block_factored_mask_is_the_decay_mask(gamma, reverse, Lc):
    M, worst = block_mask(gamma, reverse, Lc)
    assert worst >= 0                                   # every factor <= 1
    R = reference_mask(gamma, reverse, Lc)
    # rows past the end are outputs that are never stored; every key column of
    # the stored rows must match, so keys past the end must come out zero
    assert np.allclose(M[:Lc], R[:Lc], rtol=1e-12, atol=0)
