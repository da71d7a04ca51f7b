"""CPU checks of which kernel each GEMM call launches (host logic in the
library, read through wq_debug_route, the same function the entry points
dispatch on; no GPU needed):
- few tokens on the benchmark layers go to the CTA-pair decode kernel;
- 32..64 tokens go to the tensor-core kernel only when the layer has a
  128-row tile for every two SMs (the measured crossover), and 65 or more
  tokens always do;
- a route that uses the split-K workspace always has a nonzero workspace
  query, and the routes that need none have a zero query where the query
  knows it (it is an upper bound for 17..64 tokens)."""

import pytest

import weight_only_int2_gb300 as wq

K = 5120
SMS = 152


@pytest.mark.parametrize("bits", [5, 6, 7])
@pytest.mark.parametrize("N", [5120, 17408])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_sweep_takes_the_pair_kernel(M, N, bits):
    assert wq.debug_route(M, N, K, bits, SMS) == "decode_pair"


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a8_few_tokens_take_the_pair_kernel(M):
    assert wq.debug_route(M, 17408, K, 4, SMS, w4a8=True) == "decode_pair"


@pytest.mark.parametrize("M", [512, 8192])
def test_w4a8_many_tokens_take_the_tensor_cores(M):
    assert wq.debug_route(M, 17408, K, 4, SMS, w4a8=True) == "tensor_core"


def test_lm_head():
    assert wq.debug_route(1, 248320, K, 8, SMS) == "decode_pair"
    assert wq.debug_route(4096, 248320, K, 8, SMS) == "tensor_core"


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_tensor_core_crossover_at_one_tile_per_two_sms(sms):
    tiles = (sms + 1) // 2                      # the fewest 128-row tiles that qualify
    at, below = 128 * tiles, 128 * (tiles - 1)
    for M in (32, 48, 64):
        assert wq.debug_route(M, at, K, 6, sms) == "tensor_core"
        assert wq.debug_route(M, at - 127, K, 6, sms) == "tensor_core"   # a ragged last tile counts
        assert wq.debug_route(M, below, K, 6, sms) == "chunked"
    for M in (17, 24, 31):
        assert wq.debug_route(M, 17408, K, 6, sms) == "chunked"
    for M in (65, 512, 8192):
        assert wq.debug_route(M, 128, K, 6, sms) == "tensor_core"


def test_k_not_a_multiple_of_1024_streams_through_the_chunked_kernel():
    for M in (1, 16):
        assert wq.debug_route(M, 5120, 2560, 6, SMS) == "chunked"
        assert wq.debug_route(M, 5120, 2560, 4, SMS, w4a8=True) == "chunked"


@pytest.mark.parametrize("sms", [152, 132, 2])
def test_workspace_query_covers_the_route(sms):
    for M in (1, 8, 16, 17, 32, 64, 65, 4096):
        for N in (1, 1000, 5120, 17408, 248320):
            for Kx in (128, 1024, 2560, 5120, 65536):
                for bits in (2, 5, 8):
                    r = wq.debug_route(M, N, Kx, bits, sms)
                    need = wq.wna16_workspace_bytes(M, N, Kx, bits)
                    if r in ("chunked", "decode_splitk"):
                        assert need >= M * N * 4, (M, N, Kx, bits, r)
                    elif r == "decode_pair" or M >= 65:
                        assert need == 0, (M, N, Kx, bits, r)
                r4 = wq.debug_route(M, N, Kx, 4, sms, w4a8=True)
                if r4 in ("chunked", "decode_splitk"):
                    assert wq.w4a8_workspace_bytes(M, N, Kx) >= M * N * 4


@pytest.mark.parametrize("args", [
    (0, 8, 128, 6, 152, False),      # M < 1
    (1, 0, 128, 6, 152, False),      # N < 1
    (1, 8, 100, 6, 152, False),      # K not a multiple of 128
    (1, 8, 128, 9, 152, False),      # bits out of range
    (1, 8, 128, 6, 0, False),        # no SMs
    (1, 8, 128, 6, 152, True),       # W4A8 weights are 4-bit
])
def test_bad_arguments(args):
    M, N, Kx, bits, sms, w4a8 = args
    with pytest.raises(wq.WQError):
        wq.debug_route(M, N, Kx, bits, sms, w4a8=w4a8)


def test_long_k_below_the_tensor_core_token_counts():
    """Below the tensor-core kernel's token counts the chunked kernel keeps at
    most 128 groups of scales per CTA and splits a longer K over up to 64
    CTAs (K <= 1048576); a longer K has no kernel, and the entry points refuse
    it (WQ_EUNSUPPORTED) instead of failing at launch."""
    assert wq.debug_route(24, 5120, 16384, 6, SMS) == "chunked"
    assert wq.debug_route(1, 5120, 16512, 6, SMS) == "chunked"        # not a multiple of 1024
    assert wq.debug_route(24, 5120, 28672, 6, SMS) == "chunked"
    assert wq.debug_route(64, 5120, 28672, 6, SMS) == "chunked"       # too few row tiles for the tensor cores
    assert wq.debug_route(24, 5120, 28672, 4, SMS, w4a8=True) == "chunked"
    assert wq.debug_route(24, 5120, 1048576, 6, SMS) == "chunked"     # the largest K it takes
    assert wq.debug_route(24, 5120, 1048576 + 128, 6, SMS) == "none"
    assert wq.debug_route(1, 5120, 1048576 + 128, 6, SMS) == "none"
    assert wq.debug_route(64, 17408, 28672, 6, SMS) == "tensor_core"
    assert wq.debug_route(100, 5120, 28672, 6, SMS) == "tensor_core"
    assert wq.debug_route(16, 8192, 28672, 6, SMS) == "decode_splitk"


def test_zero_query_means_the_pair_kernel_on_every_device():
    """The workspace query decides 'no workspace' for a few-token shape
    without knowing the SM count: the pair plan's smallest configuration must
    fit at min(N, 256) rows, at least the largest chunk any SM count gives. So
    a zero query must mean the pair kernel at every SM count. (The converse
    may fail where that bound is not reached, e.g. 257 rows give chunks of at
    most 129: there the query is an upper bound, as documented.)"""
    sms_list = (2, 3, 16, 76, 132, 148, 152, 160, 264)
    for bits in range(2, 9):
        for M in (1, 8, 9, 16):
            for N in (1, 31, 32, 100, 256, 257, 5120, 17408, 248320):
                for K in range(1024, 32768 + 1, 1024):
                    zero = wq.wna16_workspace_bytes(M, N, K, bits) == 0
                    routes = {wq.debug_route(M, N, K, bits, sms) for sms in sms_list}
                    if zero:
                        assert routes == {"decode_pair"}, (M, N, K, bits, routes)


def test_zero_point_routes_and_workspace_query():
    """Asymmetric groups: the same kernels except the persistent split-K
    decode kernel (no zero-point mode), whose shapes the chunked kernel takes;
    the zero-point workspace query covers the need of every route it can
    take, across shapes and SM counts."""
    import random

    from weight_only_int2_gb300 import _lib as L

    lib = L.load()
    rnd = random.Random(7)
    seen = set()
    for _ in range(4000):
        M = rnd.choice([1, 2, 4, 8, 9, 16, 17, 31, 32, 48, 64, 65, 300])
        N = rnd.choice([1, 37, 300, 5120, 17408, 60000])
        K = 128 * rnd.choice([1, 5, 8, 16, 40, 56, 64, 112, 128, 136])
        bits = rnd.randint(2, 8)
        sms = rnd.choice([2, 20, 132, 148, 152])
        r = wq.debug_route(M, N, K, bits, sms, zp=True)
        seen.add(r)
        assert r != "decode_splitk"
        need = wq.wna16_zp_workspace_bytes(M, N, K, bits)
        if r == "chunked":
            assert need >= M * N * 4, (M, N, K, bits, sms)
        if r == "none":
            assert K > 1048576
        sym = wq.debug_route(M, N, K, bits, sms)
        if sym == "tensor_core":
            assert r == "tensor_core"
    assert {"decode_pair", "chunked", "tensor_core"} <= seen
    assert lib.wna16_zp_workspace_bytes(1, 17408, 5120, 6) == 0
