"""CPU checks of the CTA-pair decode kernel's launch plan (host logic in the
library, read through wq_debug_decode_plan; no GPU needed). Each invariant is
one the kernel relies on:
- ksplit divides the ring depth and the groups of a K half, so that every
  mbarrier parity wait is on a phase whose predecessor the waiter consumed;
- TMA boxes stay within the hardware limits (256 rows; 16-byte-multiple
  rows and x coordinates for the scale box);
- the scale box of each K half covers that half's groups;
- the clusters' chunks cover every output row, and the warps fit in a CTA;
- the shared-memory carve-up fits the 227 KB a CTA may use."""

import pytest

import weight_only_int2_gb300 as wq

SMEM_CAP = 227 * 1024


def _rows(N, C, cid):
    return (cid + 1) * N // C - cid * N // C


@pytest.mark.parametrize("sms", [152, 148, 132, 16, 2])
@pytest.mark.parametrize("bits", range(2, 9))
def test_plan_invariants(bits, sms):
    n_ok = 0
    for K in (1024, 2048, 4096, 5120, 8192, 16384, 31744):
        for N in (1, 31, 32, 33, 100, 1000, 5120, 17408, 248320, 1 << 20):
            for M in (1, 2, 5, 8, 9, 16):
                p = wq.debug_decode_plan(M, N, K, bits, sms)
                if not p["ok"]:
                    continue
                n_ok += 1
                assert 1 <= M <= 16 and K % 1024 == 0
                assert p["G"] == K // 128 and p["Gh"] == p["G"] // 2
                assert p["NT"] == (1 if M <= 8 else 2)
                assert 1 <= p["C"] <= sms // 2 and p["C"] <= -(-N // 32)
                assert 1 <= p["H"] <= 256 and p["T"] == -(-p["H"] // 32)
                assert max(_rows(N, p["C"], c) for c in (0, p["C"] - 1)) <= p["nchunk"] * p["H"]
                assert p["T"] * p["ksplit"] <= 16
                assert p["Gh"] % p["ksplit"] == 0 and p["NS"] % p["ksplit"] == 0
                assert 2 <= p["NS"] <= p["max_slots"]
                assert p["sbox"] % 8 == 0 and p["sx0"] % 8 == 0 and p["sbox"] <= 256
                assert p["sbox"] >= p["Gh"]                                   # half 0: [0, Gh)
                assert p["sx0"] <= p["Gh"] and p["sx0"] + p["sbox"] >= p["G"]  # half 1: [Gh, G)
                assert 0 < p["smem"] <= SMEM_CAP
    if sms >= 16:
        assert n_ok > 0


@pytest.mark.parametrize("bits", [5, 6, 7])
@pytest.mark.parametrize("N", [5120, 17408])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_benchmark_shapes_use_the_pair_kernel(bits, N, M):
    assert wq.debug_decode_plan(M, N, 5120, bits, 152)["ok"] == 1


def test_lm_head_shape_is_chunked():
    p = wq.debug_decode_plan(1, 248320, 5120, 8, 152)
    assert p["ok"] == 1 and p["nchunk"] > 1


@pytest.mark.parametrize("args", [(1, 1000, 5000, 6, 152), (17, 1000, 5120, 6, 152), (0, 1000, 5120, 6, 152),
                                  (1, 1000, 512, 6, 152)])
def test_unsupported_shapes_are_refused(args):
    assert wq.debug_decode_plan(*args)["ok"] == 0


def test_bad_arguments():
    with pytest.raises(wq.WQError):
        wq.debug_decode_plan(1, 1000, 5120, 9, 152)
    with pytest.raises(wq.WQError):
        wq.debug_decode_plan(1, 1000, 5120, 6, 0)
