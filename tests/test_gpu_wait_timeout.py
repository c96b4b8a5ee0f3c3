"""The device-side failure path: a bounded wait that runs out (q8_selftest_wait_timeout).

The self-test runs a kernel whose TMA producer issues no load, so the converter (decode:
compute) warps' wait on the first stage can never complete; with a short limit it gives up,
records which wait it was in the device error word and winds the kernel down with nothing
in flight. The host reads Q8_ERR_TIMEOUT through q8_device_error, and the next normal call
on the same process (for the tcgen05 kernel: the next allocation of tensor memory on the
same SMs) must run and be bit-exact. No GPU fault is involved: the failure is a wait that
nothing satisfies, and every wait in the kernels is bounded.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SHORT_WAIT = 1 << 24          # clock cycles (~8 ms at 2 GHz)


@pytest.fixture(scope="module")
def q8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import int8_quantized_gemm_gb300 as q8mod
    from int8_quantized_gemm_gb300 import build
    build.build()
    q8mod.load()
    return q8mod


def codes(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    return qa, qw


@pytest.mark.parametrize("kernel,M,N,K,code", [
    ("decode", 16, 128, 512, 2 << 16),      # decode kernel: the compute warps' wait on a loaded stage
    ("tcgen05", 256, 512, 1024, 2),         # single-CTA tcgen05 kernel: the converters' wait
])
def test_wait_runs_out_and_the_next_call_is_exact(q8, kernel, M, N, K, code):
    qa, qw = codes(M, N, K, seed=M + N)
    qa_d, qw_d = torch.from_numpy(qa).cuda(), torch.from_numpy(qw).cuda()
    assert q8.q8_device_error() == 0
    acc = q8.q8_selftest_wait_timeout(qa_d, qw_d, kernel=kernel, wait_cycles=SHORT_WAIT)
    torch.cuda.synchronize()                      # the kernel returned: no hang, no CUDA error
    assert q8.q8_device_error() == code           # Q8_ERR_TIMEOUT with that role's bit
    assert q8.q8_device_error() == 0              # reading the word resets it
    assert int(acc.abs().max()) == 0              # the aborted kernel wrote nothing
    ref = oracle.gemm_acc(qa, qw)
    for _ in range(2):                            # the same kernel again, normally: bit-exact
        got = q8.q8_gemm_s32(qa_d, qw_d, kernel=kernel)
        torch.cuda.synchronize()
        assert q8.q8_device_error() == 0
        np.testing.assert_array_equal(got.cpu().numpy().astype(np.int64), ref)


def test_selftest_rejects_bad_arguments(q8):
    qa = torch.zeros((16, 64), dtype=torch.int8, device="cuda")
    qw = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    for kernel, cycles in (("tcgen05_pair", SHORT_WAIT), ("decode", 0), ("decode", (1 << 31) + 1)):
        with pytest.raises(q8.Q8Error) as e:
            q8.q8_selftest_wait_timeout(qa, qw, kernel=kernel, wait_cycles=cycles)
        assert e.value.status == q8.Q8_ERR_INVALID_ARG
    assert q8.q8_device_error() == 0
