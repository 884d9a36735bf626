"""GPU checks of the peak probes (include/gemm_probe.h): they run, leave the
device status clean, and report rates that a working probe can reach -- well
above a broken or serialised kernel, and not above what the SM count and the
maximum clock allow (a count of FLOPs that the kernel does not perform would
show up as a rate above the ceiling)."""
import pytest
import torch

import dense_gemm_08_gb300 as lib

pytestmark = pytest.mark.gpu


def _rate(launch, reps=3):
    stream = torch.cuda.current_stream()
    launch()
    torch.cuda.synchronize()
    best = 0.0
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st, flops = launch()
        e1.record(stream)
        e1.synchronize()
        assert st == lib.GEMM_OK
        best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    return best


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("cta_group", [1, 2])
def test_tensor_probe_rate_is_plausible(cta_group):
    flops_per_mma = 2.0 * 128 * cta_group * 256 * 16
    st, flops = lib.gemm_probe_tc_bf16(cta_group, 1000)
    assert st == lib.GEMM_OK and flops > 0
    groups = flops / (flops_per_mma * 1000)
    assert groups == int(groups) and 1 <= groups <= _sms() / cta_group
    tflops = _rate(lambda: lib.gemm_probe_tc_bf16(cta_group, 20000))
    # ceiling: 8192 dense BF16 FLOPs per SM per clock at 2.1 GHz
    ceiling = _sms() * 8192 * 2.1e9 / 1e12
    assert 300.0 < tflops < 1.05 * ceiling, tflops
    assert lib.gemm_last_kernel().startswith("tc_probe")


def test_fma_probe_rate_is_plausible():
    tflops = _rate(lambda: lib.gemm_probe_fma_f32(2000))
    ceiling = _sms() * 128 * 2 * 2.1e9 / 1e12  # 128 FP32 lanes per SM at 2.1 GHz
    assert 0.3 * ceiling < tflops < 1.02 * ceiling, tflops
    assert lib.gemm_last_kernel() == "fma_probe"


def test_probe_leaves_gemm_results_intact():
    # a GEMM after the probes still matches a plain CPU product exactly
    # (small integers: every partial sum is exact in FP32)
    lib.gemm_probe_tc_bf16(2, 500)
    lib.gemm_probe_fma_f32(100)
    g = torch.Generator().manual_seed(7)
    a = torch.randint(-4, 5, (300, 200), generator=g).to(torch.bfloat16)
    b = torch.randint(-4, 5, (200, 500), generator=g).to(torch.bfloat16)
    d = lib.gemm(a.cuda(), b.t().contiguous().cuda().t())
    ref = a.double() @ b.double()
    assert torch.equal(d.cpu().double(), ref)


def test_bounded_wait_gives_up_and_reports_timeout():
    """The failure path without a broken kernel: a wait on a barrier nothing
    completes gives up after 5 ms, the status word says GEMM_ERR_TIMEOUT once,
    and the context stays usable (a GEMM afterwards is exact)."""
    import time
    assert lib.gemm_last_device_status() == lib.GEMM_OK
    t0 = time.perf_counter()
    assert lib.gemm_probe_wait_timeout(5_000_000) == lib.GEMM_OK
    assert lib.gemm_last_kernel() == "wait_probe"
    assert lib.gemm_last_device_status() == lib.GEMM_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert lib.gemm_last_device_status() == lib.GEMM_OK  # read and cleared
    test_probe_leaves_gemm_results_intact()
