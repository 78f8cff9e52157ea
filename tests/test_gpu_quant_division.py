"""The quantizer's division by a scale against the IEEE float32 quotient (GPU).

The fp8 and NVFP4 rules round the float32 quotient x / s of an fp16 value by a
float32 scale (and NVFP4's block-scale rule rounds max|x| / RN(6 s)).  The
quantizer computes that quotient from RN(1 / s) with two exact-remainder
refinements instead of an IEEE division; here it must equal __fdiv_rn in every
bit, for every finite fp16 dividend, over the scales the rules produce and
scales spread across the float32 range.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def memra():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_attention_block_memra_gb300 import _build
    _build.build()
    import decode_attention_block_memra_gb300 as m
    m.lib()
    return m


def _scales():
    f32 = np.float32
    pos16 = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float32)   # finite fp16 > 0
    e4m3 = torch.arange(1, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()   # finite e4m3 > 0
    fp8_tensor = (pos16 / f32(448.0)).astype(f32)                  # per-tensor fp8 scales amax / 448
    nv_tensor = (pos16[::257] / f32(2688.0)).astype(f32)           # NVFP4 tensor scales amax / (6 * 448)
    nv_block = (e4m3[None, :] * nv_tensor[:, None]).astype(f32).ravel()       # e4m3 block scale x tensor scale
    nv_six = (f32(6.0) * nv_tensor).astype(f32)                    # the block-scale rule's divisor RN(6 s)
    pow2 = np.ldexp(f32(1.0), np.arange(-70, 71)).astype(f32)     # both sides of the [2^-60, 2^60] range
    edges = np.array([np.nextafter(f32(2.0 ** -60), f32(0)), np.nextafter(f32(2.0 ** -60), f32(1)),
                      np.nextafter(f32(2.0 ** 60), f32(0)), np.nextafter(f32(2.0 ** 60), f32(np.inf))], f32)
    rng = np.random.default_rng(17)
    spread = np.exp2(rng.uniform(-60, 60, 20000)).astype(f32)
    mant = (f32(1.0) + rng.integers(0, 1 << 23, 4000).astype(f32) * f32(2.0 ** -23)).astype(f32)
    near_one = (mant * np.ldexp(f32(1.0), rng.integers(-8, 9, 4000))).astype(f32)
    return np.concatenate([fp8_tensor, nv_block, nv_six, pow2, edges, spread, near_one]).astype(np.float32)


def test_division_free_quotient_equals_ieee(memra):
    scales = _scales()
    assert (scales > 0).all() and np.isfinite(scales).all()
    mism = torch.zeros(1, dtype=torch.int64, device="cuda")
    s_dev = torch.from_numpy(scales).cuda()
    for i in range(0, scales.size, 65535):
        memra.testing_scale_division_mismatches(s_dev[i:i + 65535], mism)
    torch.cuda.synchronize()
    assert int(mism.item()) == 0, f"{int(mism.item())} of {scales.size} x 63,488 quotients differ"
