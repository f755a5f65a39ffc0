"""The parity metric on the CPU: per (sequence, head) slice, max|x - ref| /
max|ref|, the worst slice deciding; NaN fails; the failure message carries the
RMS-relative error too."""
import numpy as np
import pytest

from parity import compare, rms_rel, slice_err


def _pair(seed=0):
    rng = np.random.default_rng(seed)
    ref = rng.standard_normal((2, 40, 3, 8))
    ref[:, :, 0] *= 1e4            # a head whose values grow large (zero decay)
    return ref


def test_a_large_head_does_not_hide_a_small_heads_error():
    ref = _pair()
    got = ref.copy()
    got[1, 7, 2, 3] += 0.05 * np.abs(ref[1, :, 2]).max()     # 5 % in a small head
    assert abs(slice_err(got, ref) - 0.05) < 1e-12
    # the whole-tensor ratio would see almost nothing
    assert np.abs(got - ref).max() / np.abs(ref).max() < 1e-4


def test_packed_slices_and_states():
    ref = _pair()[:1]
    got = ref.copy()
    cu = [0, 10, 10, 40]                                        # an empty sequence too
    got[0, 12, 1, 0] += 0.01 * np.abs(ref[0, 10:40, 1]).max()
    assert abs(slice_err(got, ref, cu) - 0.01) < 1e-12
    st = np.ones((3, 2, 4, 4))
    st2 = st.copy()
    st2[2, 1, 0, 0] = 1.5
    assert abs(slice_err(st2, st, state=True) - 0.5) < 1e-12


def test_compare_fails_on_nan_and_reports_rms():
    ref = _pair()
    got = ref.copy()
    got[0, 0, 1, 0] = np.nan
    with pytest.raises(AssertionError, match="RMS-relative"):
        compare({"o": got}, {"o": ref}, 2e-2, label="nan")
    assert compare({"o": ref + 1e-9}, {"o": ref}, 2e-2)["o"] < 1e-8
    assert rms_rel(ref * 1.01, ref) == pytest.approx(0.01)
