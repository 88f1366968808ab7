"""GPU tests of gdr_check_cu_seqlens, the opt-in device-side check of the
packed-sequence contract (cu[0] = 0, non-decreasing, cu[B] <= T).

Only the check kernel ever sees a broken array: it reads cu[0..B] and nothing
else, so a broken array causes no fault; the solve itself only runs on valid
arrays here.  Varlen bookkeeping is where the MindSpeed-Ops PR #135 page's own
fix landed (bot summary: the T_local fix), hence a check a caller can switch on.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _status_after_check(cu, T, dev):
    gdr.check_cu_seqlens(torch.tensor(cu, dtype=torch.int32, device=dev), T)
    return gdr.device_status()


@pytest.mark.parametrize("cu,T", [
    ([0], 0), ([0], 5), ([0, 0], 0), ([0, 5], 5), ([0, 5], 9), ([0, 3, 3, 70, 200], 200),
    ([0, 1, 65, 65, 130, 258, 260, 323, 523, 523, 652], 700)])
def test_valid_arrays_pass(cu, T):
    dev = _dev()
    assert gdr.device_status() == gdr.GDR_OK
    assert _status_after_check(cu, T, dev) == gdr.GDR_OK


@pytest.mark.parametrize("cu,T", [
    ([1, 5], 9),                 # cu[0] != 0
    ([0, 5, 4, 9], 9),           # decreasing step
    ([0, 5, 10], 9),             # cu[B] > T
    ([-3, 5], 9),                # negative start
    ([0, -1, 4], 9),             # negative inside
    ([0, 2 ** 31 - 1, 7], 10),   # huge then smaller
])
def test_broken_arrays_are_reported_without_a_fault(cu, T):
    dev = _dev()
    assert gdr.device_status() == gdr.GDR_OK
    assert _status_after_check(cu, T, dev) == gdr.GDR_ERR_CU_SEQLENS
    # Reading the status cleared it; the context is usable and the next check is clean.
    assert gdr.device_status() == gdr.GDR_OK
    assert _status_after_check([0, 4, 9], 9, dev) == gdr.GDR_OK


def test_many_sequences_every_position_is_checked():
    # 300001 entries: the grid-stride loop covers all of them; one swapped pair
    # anywhere is found.
    dev = _dev()
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 9, size=300000)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    assert _status_after_check(cu.tolist(), T, dev) == gdr.GDR_OK
    for pos in (1, 150000, 299999):
        bad = cu.copy()
        bad[pos] = bad[pos + 1] + 1
        assert _status_after_check(bad.tolist(), T + 1, dev) == gdr.GDR_ERR_CU_SEQLENS, pos
    assert gdr.device_status() == gdr.GDR_OK


def test_an_earlier_unread_status_is_kept():
    dev = _dev()
    assert gdr.selftest_bounded_wait(torch.cuda.current_stream(dev).cuda_stream) == gdr.GDR_OK
    gdr.check_cu_seqlens(torch.tensor([1, 5], dtype=torch.int32, device=dev), 9)
    assert gdr.device_status() == gdr.GDR_ERR_TIMEOUT
    assert gdr.device_status() == gdr.GDR_OK


def test_validated_call_equals_the_plain_call():
    dev = _dev()
    wl = workloads.CONFIGS["varlen8_H16_K128"]
    inp = workloads.make_inputs(wl)
    k, g, b, cu = (inp[x].to(dev) for x in ("k", "g", "beta", "cu_seqlens"))
    plain = gdr.kkt_solve(k, g, b, cu, output_dtype=torch.float32)
    checked = gdr.kkt_solve(k, g, b, cu, output_dtype=torch.float32, validate_cu_seqlens=True)
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    assert torch.equal(plain, checked)
