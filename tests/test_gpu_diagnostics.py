"""The diagnostics: the bounded-wait expiry path and the HBM read probe, on the GPU.

The wait-expiry check runs the kernels' own bounded mbarrier wait on a phase that
nothing completes, with a short bound (a few thousand polls): the timeout must
reach q4lin_device_status(), the kernel must return (no hang, no fault), and the
same context must still compute the layer correctly afterwards.
"""
import numpy as np
import pytest

import oracle
from weight_only_bit_q4_gb300 import q4lin, synth

from gpu_util import assert_close, to_dev, torch, y_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from weight_only_bit_q4_gb300 import build
    build.build()
    q4lin.load()
    yield


def test_wait_expiry_reports_timeout_and_context_stays_usable():
    t = torch()
    assert q4lin.clear_device_status() == 0
    assert q4lin.device_status() == 0
    out = t.full((1,), -1, dtype=t.int32, device="cuda")
    q4lin.diag_wait_expiry(4096, out)
    t.cuda.synchronize()
    assert int(out.item()) == 2            # the wait did not succeed and the abort flag is up
    assert q4lin.device_status() == 7      # Q4LIN_ERR_TIMEOUT, sticky until cleared
    assert q4lin.device_status() == 7
    assert q4lin.clear_device_status() == 0
    assert q4lin.device_status() == 0
    # the context still runs the layer: one call per route family, checked against the oracle
    for (N, K, T) in [(512, 1024, 8), (6144, 5120, 1), (640, 2048, 300)]:
        wq, s, x = synth.make_problem(N, K, T, w_seed=11, x_seed=12)
        y = q4lin.linear(*to_dev(wq, s, x))
        t.cuda.synchronize()
        assert_close(y_bits(y), oracle.linear(wq, s, x), f"{N}x{K} T={T} after a timeout")
    assert q4lin.device_status() == 0


def test_wait_expiry_rejects_bad_bounds():
    t = torch()
    out = t.zeros((1,), dtype=t.int32, device="cuda")
    for bad in (0, (1 << 20) + 1):
        with pytest.raises(q4lin.Q4LinError):
            q4lin.diag_wait_expiry(bad, out)


@pytest.mark.parametrize("nbytes,blocks", [(16, 1), (4096 + 16, 3), ((64 << 20) + 48, 0)])
def test_hbm_read_probe_reads_every_word_once(nbytes, blocks):
    t = torch()
    rng = np.random.default_rng(nbytes)
    words = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = t.from_numpy(words.view(np.int32)).cuda()
    nb = blocks if blocks > 0 else 4 * t.cuda.get_device_properties(0).multi_processor_count
    sink = t.zeros((nb,), dtype=t.int32, device="cuda")
    q4lin.hbm_read_probe(buf, sink, blocks)
    t.cuda.synchronize()
    got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
    assert got == np.bitwise_xor.reduce(words)
