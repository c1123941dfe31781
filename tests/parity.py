"""The element bound of the GPU parity tests, kept free of torch so the CPU tests can exercise it.

Every output element o (bf16) of (row r, head h) is held to

    |o - o64| <= 2^-8 |o64| + c * rms_h(o64)

where o64 is the oracle's f64 value and rms_h(o64) = sqrt(mean_d o64[r, h, d]^2) is the
RMS of that (row, head)'s output.  The two terms follow the arithmetic of the kernels:

* output rounding: o is o64's f32 accumulation rounded to nearest bf16, at most half an
  ulp, 2^-9 |o|; the first term allows twice that;
* rounding of the probabilities: every P value is rounded to bf16 (relative error up to
  2^-9) and the row's sum is taken from the same rounded values, so the output moves by
  sum_t w_t delta_t (v_t - o): a sum of independent rounding errors weighted like the
  output itself.  For the zero-mean V of most workloads its standard deviation is about
  0.6 * 2^-9 * rms_h(o64), and over up to ~3e7 elements it stays below about
  3 * 2^-9 = 2^-7.4 rms_h -- hence c = 2^-7 for the decode kernel and the hd-512 prefill
  (mma.sync, P in [0, 1]).  The tcgen05 kernels let P grow to 2^8 before rescaling O and
  accumulate 64-token blocks inside the tensor core, which doubles that: c = 2^-6.

A (row, head) with no visible position has o64 = 0 and must be exactly zero.

Beside it, the whole output's rel-RMS against the f64 values (not against the oracle's
truncated bf16, whose own truncation already costs about 4e-3 of the page's 1e-2 gate)
must stay below 2^-8: round-to-nearest output alone contributes about 2^-9 / sqrt(3)
relative, the rounding of P about half that again.  A mask one token off over 32K
positions moves it to about 6e-3.
"""
import numpy as np

COEF_DECODE = 2.0 ** -7
COEF_TILED = 2.0 ** -6
REL_RMS_F64_GATE = 2.0 ** -8


def bf16_bits_to_f64(b):
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def element_bound(ref64, coef=COEF_DECODE):
    """Per-element bound, shaped like ref64 ([..., hd])."""
    r = np.asarray(ref64, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    return 2.0 ** -8 * np.abs(r) + coef * rms


def beyond_bound(got_bits, ref64, coef=COEF_DECODE):
    """Boolean mask of the elements of got (bf16 bits) beyond the bound (NaN counts as beyond)."""
    g = bf16_bits_to_f64(got_bits).reshape(np.shape(ref64))
    d = np.abs(g - ref64)
    return ~(d <= element_bound(ref64, coef))


def rel_rms_f64(got_bits, ref64):
    """sqrt(sum (o - o64)^2 / sum o64^2) against the oracle's f64 values (not its truncated bf16)."""
    g = bf16_bits_to_f64(got_bits).reshape(np.shape(ref64))
    den = float(np.sum(np.asarray(ref64) ** 2))
    return float(np.sqrt(float(np.sum((g - ref64) ** 2)) / max(den, 1e-30)))
