"""GPU index maps (shard ownership, tile classes, element masks) bit-exact
against the oracle's plain enumeration, and the bounded-wait error path."""
import numpy as np
import pytest
import torch

from oracle import shardmap as OS

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("N,P", [(8, 4), (12, 3), (4096, 16), (1 << 20, 64), (96, 96)])
def test_device_shard_map_bit_exact(layout, N, P):
    if layout == "zigzag" and N % (2 * P):
        # zigzag needs N divisible by 2P: refused before any launch
        with pytest.raises(ra.RingAttnError, match="RA_ERR_INVALID_ARG"):
            ra.shard_map_device(layout, N, P, DEV)
        return
    own, loc, tok = ra.shard_map_device(layout, N, P, DEV)
    torch.cuda.synchronize()
    if N <= 4096:
        w_own, w_loc, w_tok = OS.shard_map(layout, N, P)
    else:   # the oracle's formulas, vectorised for the 1M-token map
        t = np.arange(N)
        S = N // P
        w_own = [OS.owner(layout, N, P, int(x)) for x in t[:: 997]]
        w_loc = [OS.local_index(layout, N, P, int(x)) for x in t[:: 997]]
        w_tok = [OS.token_of(layout, N, P, int(x) // S, int(x) % S) for x in t[:: 997]]
        own, loc, tok = own[:: 997], loc[:: 997], tok[:: 997]
        # and the full maps are inverse permutations
        o_all, l_all, k_all = (x.cpu().numpy() for x in ra.shard_map_device(layout, N, P, DEV))
        assert np.array_equal(np.sort(k_all), t)
        assert np.array_equal(k_all[o_all * S + l_all], t)
    assert own.cpu().tolist() == list(w_own)
    assert loc.cpu().tolist() == list(w_loc)
    assert tok.cpu().tolist() == list(w_tok)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,P", [(4 * 300, 4), (3 * 128, 3), (2 * 40, 2), (4 * 176, 2)])
def test_tile_classes_bit_exact(layout, causal, N, P):
    pr = ra.problem(1, N, 1, 1, 128, P, causal, layout)
    for u in range(P):
        for b in range(P):
            got = ra.tile_classes(pr, u, b, DEV).cpu().tolist()
            want = OS.tile_classes(layout, N, P, causal, u, b, ra.TILE, ra.TILE)
            assert got == want, (u, b)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("N,P", [(8 * 37, 4), (5 * 20, 5)])
def test_element_mask_bit_exact(layout, N, P):
    pr = ra.problem(1, N, 1, 1, 64, P, True, layout)
    for u in range(P):
        for b in range(P):
            got = ra.mask(pr, u, b, DEV).cpu().numpy().astype(bool)
            want = np.array(OS.mask_block(layout, N, P, True, u, b), dtype=bool)
            assert np.array_equal(got, want), (u, b)


def test_bounded_wait_reports_timeout_and_context_survives():
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    ra.selftest_timeout(2_000_000, DEV)           # 2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == ra.RA_ERR_TIMEOUT
    assert ra.last_error(DEV) == 0                 # reading clears it
    # the context is still usable
    x = torch.ones(16, device=DEV)
    assert float(x.sum()) == 16.0
