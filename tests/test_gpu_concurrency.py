"""Calls on several CUDA streams at once, and from several host threads at
once (each with its own stream), give the results of the same calls made one
after another: the kernels keep no state between calls beyond the
zero-at-rest workspaces (one per caller here), and the host side's shared
tables (encoded TMA descriptors, shared-memory limits) are locked. Routes
that reduce in a fixed order must give the same bits; the split-K streaming
routes add their partial sums with fp32 atomics (any order), so theirs are
compared within a bf16 rounding of the sequential result."""

import threading

import numpy as np
import pytest

import wq_inputs as I
from helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402

K = 2048


def _jobs(seed):
    """A mix of routes: pair decode, tensor-core prefill, split-K streaming,
    W4A8 one-launch decode, and the gather."""
    rng = np.random.default_rng(seed)
    jobs = []
    for (M, N, bits) in ((1, 2048, 6), (16, 1536, 5), (200, 1024, 7), (24, 768, 4)):
        q = I.make_codes(N, K, bits, int(rng.integers(1 << 30)))
        s = I.make_scales(N, K // 128, int(rng.integers(1 << 30)))
        packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
        x = to_dev_bf16(I.make_x(M, K, int(rng.integers(1 << 30))))
        ws = torch.zeros(max(1, wq.wna16_workspace_bytes(M, N, K, bits)), dtype=torch.uint8, device="cuda")
        jobs.append(("wna16", x, packed, s_dev, N, bits, ws))
    q4 = I.make_codes(1024, K, 4, int(rng.integers(1 << 30)))
    s4 = I.make_scales(1024, K // 128, int(rng.integers(1 << 30)))
    p4, sd4 = wq.wna16_repack(to_dev(q4), to_dev_bf16(s4), 4)
    jobs.append(("w4a8", to_dev_bf16(I.make_x_outliers(2, K, int(rng.integers(1 << 30)))), p4, sd4, 1024, 4, None))
    ids = torch.from_numpy(rng.integers(0, 1024, size=64).astype(np.int32)).cuda()
    jobs.append(("gather", ids, p4, sd4, 1024, 4, None))
    return jobs


def _run(job):
    kind, a, packed, s_dev, N, bits, ws = job
    if kind == "wna16":
        return wq.wna16_gemm(a, packed, s_dev, N, K, bits, ws=ws)
    if kind == "w4a8":
        return wq.w4a8_gemm(a, packed, s_dev, N, K)
    return wq.qembed_gather(a, packed, s_dev, N, K, bits)


def _bits(t):
    return t.view(torch.int16).clone()


def _deterministic(job):
    kind, a, packed, s_dev, N, bits, ws = job
    if kind != "wna16":
        return True
    return wq.debug_route(a.shape[0], N, K, bits, torch.cuda.get_device_properties(0).multi_processor_count) in (
        "decode_pair", "tensor_core")


def _same(job, y, ref_bits, what):
    if _deterministic(job):
        assert torch.equal(y.view(torch.int16), ref_bits), what
    else:
        ref = ref_bits.view(torch.bfloat16).float()
        err = (y.float() - ref).abs().max().item()
        assert err <= 2 ** -7 * ref.abs().max().item(), (what, err)


def test_streams_run_concurrently_with_identical_results():
    sets = [_jobs(8100 + i) for i in range(3)]
    ref = [[_bits(_run(j)) for j in js] for js in sets]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in sets]
    outs = [[] for _ in sets]
    for rep in range(10):
        for si, (st, js) in enumerate(zip(streams, sets)):
            with torch.cuda.stream(st):
                outs[si].append([_run(j) for j in js])
    torch.cuda.synchronize()
    for si in range(len(sets)):
        for rep in range(10):
            for ji, y in enumerate(outs[si][rep]):
                _same(sets[si][ji], y, ref[si][ji], (si, rep, ji))
    wq.check_status()


def test_host_threads_call_concurrently_with_identical_results():
    sets = [_jobs(8200 + i) for i in range(4)]
    ref = [[_bits(_run(j)) for j in js] for js in sets]
    torch.cuda.synchronize()
    errors = []
    results = [None] * len(sets)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            got = []
            with torch.cuda.stream(st):
                for _ in range(10):
                    got.append([_run(j) for j in sets[i]])
            st.synchronize()
            results[i] = got
        except Exception as e:  # pragma: no cover - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(sets))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, got in enumerate(results):
        for rep, ys in enumerate(got):
            for ji, y in enumerate(ys):
                _same(sets[i][ji], y, ref[i][ji], (i, rep, ji))
    wq.check_status()
