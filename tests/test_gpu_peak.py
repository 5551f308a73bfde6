"""attn_tensor_peak, the tensor-pipe rate measurement the bench's tf32
roofline uses: a short launch of each shape finishes without a device error,
and a longer one runs at a plausible rate (between a tenth and one and a half
times the nominal dense rate of its kind at the maximum clock)."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as m
    return m


@pytest.mark.parametrize("bf16,n", [(0, 64), (0, 128), (0, 256), (1, 128), (1, 256)])
def test_short_launch_completes(cp, bf16, n):
    flops = cp.attn_tensor_peak(bool(bf16), n, 64, 4)
    torch.cuda.synchronize()
    assert cp.attn_get_device_error() == 0
    assert flops == 4 * 64 * 2 * 128 * n * (16 if bf16 else 8)


@pytest.mark.parametrize("bf16", [0, 1])
def test_rate_is_plausible(cp, bf16):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    iters = 20000
    cp.attn_tensor_peak(bool(bf16), 256, iters, sms)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    flops = cp.attn_tensor_peak(bool(bf16), 256, iters, sms)
    b.record()
    torch.cuda.synchronize()
    assert cp.attn_get_device_error() == 0
    tflops = flops / (a.elapsed_time(b) * 1e-3) / 1e12
    # nominal dense flop per clock per SM at M = 128: 8192 (bf16), 4096 (tf32)
    nominal = sms * (8192 if bf16 else 4096) * 2.07e9 / 1e12
    print(f"{'bf16' if bf16 else 'tf32'} N=256: {tflops:.1f} TFLOP/s (nominal at 2.07 GHz {nominal:.0f})")
    assert 0.1 * nominal < tflops < 1.5 * nominal
