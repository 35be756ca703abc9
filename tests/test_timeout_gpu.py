"""The bounded device waits: a wait that runs out records LLA_ERR_TIMEOUT, the kernel returns, and
the stream and device stay usable.

Every mbarrier wait of the tensor-core kernels gives up after a time limit (about 2 s), sets the
timeout bit of the device status word and makes its CTA return early, after the tensor-core work
that it did issue has completed and before its tensor memory is released. The test-only fault
LLA_FAULT_WITHHOLD_KEYS (lla_forward_ex, tensor-core moments stage) makes the key loader skip its
first key block, so the waits on that block run out; nothing faults, traps or spins unbounded.
"""
import time

import numpy as np
import pytest

from local_linear_attention_gb300 import workloads as W
from oracle import lla_forward_oracle
from parity import record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lla():
    from local_linear_attention_gb300 import binding, build
    build.build()
    return binding


def test_withheld_keys_time_out_and_the_stream_stays_usable(lla):
    # one CTA pair (T = 256 queries of one head)
    q, k, v = (t.cuda() for t in W.make_iid(1, 1, 256, 64, 64, "bf16", seed=90))
    assert lla.lla_stream_status() == 0
    t0 = time.perf_counter()
    lla.lla_forward(q, k, v, 8.0, 1e-2, test_fault=lla.FAULT_WITHHOLD_KEYS)
    st = lla.lla_stream_status()
    elapsed = time.perf_counter() - t0
    assert st == 5, lla.lla_status_string(st)  # LLA_ERR_TIMEOUT
    assert elapsed < 60.0
    assert lla.lla_stream_status() == 0  # the read cleared it
    # the next call on the same stream is correct
    qc, kc, vc = W.make_iid(1, 2, 300, 64, 64, "bf16", seed=91)
    out = lla.lla_forward(qc.cuda(), kc.cuda(), vc.cuda(), 8.0, 1e-2)
    assert lla.lla_stream_status() == 0
    got = out.float().cpu().numpy().astype(np.float64).reshape(-1, 64)
    ref = lla_forward_oracle(qc, kc, vc, 8.0, 1e-2).reshape(-1, 64)
    record(got, ref, vc.float().numpy(), 2e-2)


def test_fault_needs_the_tensor_core_moments(lla):
    # fp32 inputs, and bf16 on the CUDA-core path, have no tensor-core moments stage
    q, k, v = (t.cuda() for t in W.make_iid(1, 1, 64, 32, 32, "f32", seed=92))
    with pytest.raises(lla.LlaError) as ei:
        lla.lla_forward(q, k, v, 8.0, 1e-2, test_fault=lla.FAULT_WITHHOLD_KEYS)
    assert ei.value.status == 2  # LLA_ERR_UNSUPPORTED
    q, k, v = (t.cuda() for t in W.make_iid(1, 1, 64, 32, 32, "bf16", seed=92))
    with pytest.raises(lla.LlaError) as ei:
        lla.lla_forward(q, k, v, 8.0, 1e-2, test_fault=lla.FAULT_WITHHOLD_KEYS,
                        path=lla.PATH_CUDA_CORE)
    assert ei.value.status == 2
