"""Storage rounding for the oracle (test infrastructure only).

The KV cache of [TSD-V4] §4.2 holds compressed entries in the cache's storage dtype.  The
oracle computes every entry in fp64 and then rounds it once, directly from fp64, to the
storage dtype with round-to-nearest, ties-to-even:

* ``"bf16"``: 1 sign bit, 8 exponent bits, 7 stored mantissa bits;
* ``"f32"``:  IEEE binary32;
* ``"f64"``:  no rounding (used by the brute-force self-checks).

The bf16 rounding is done on the fp64 bit pattern (drop the 45 low mantissa bits with
round-half-even), so it is a single rounding, not fp64 -> fp32 -> bf16.
"""

import numpy as np

_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_MAX = float(np.float64(np.uint64(0x47EFE00000000000).view(np.float64)))  # (2 - 2^-7) * 2^127


def to_f64(x):
    """Exact conversion of a stored array (fp32 or fp64, or bf16 already widened) to fp64."""
    return np.asarray(x, dtype=np.float64)


def _round_f64_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    ax = np.abs(x)
    if np.any(~np.isfinite(x)):
        raise ValueError("bf16 rounding: non-finite input")
    if np.any((ax != 0.0) & (ax < _BF16_MIN_NORMAL)):
        raise ValueError("bf16 rounding: value in the bf16 subnormal range")
    bits = x.view(np.uint64)
    keep_lsb = (bits >> np.uint64(45)) & np.uint64(1)
    half_minus_one = np.uint64((1 << 44) - 1)
    low_mask = np.uint64((1 << 45) - 1)
    rounded = (bits + half_minus_one + keep_lsb) & ~low_mask
    out = rounded.view(np.float64)
    if np.any(np.abs(out) > _BF16_MAX):
        raise ValueError("bf16 rounding: overflow")
    return out


def round_to_storage(x, store):
    """Round fp64 values to the storage dtype ``store`` and return them as fp64."""
    x = np.asarray(x, dtype=np.float64)
    if store == "f64":
        return x.copy()
    if store == "f32":
        return x.astype(np.float32).astype(np.float64)
    if store == "bf16":
        return _round_f64_to_bf16(x)
    raise ValueError(f"unknown storage dtype {store!r}")
