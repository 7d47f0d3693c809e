"""FP8 (E4M3) inputs for the attention oracle — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
use this module; the library never does.

"Fused Multi-Head Attention" (inferensys.com glossary), in its list of what
fused attention combines with (the "Quantization" item), says fused kernels
can take FP8 data for both GEMMs; "Kernel Fusion and the Memory Wall", the
paragraph after "A small executable reference", names low-precision
facilities as part of FlashAttention-3.  Neither page fixes a format or a
scaling rule.  Plainest reading, used here: the inputs are E4M3 codes (the
OCP 8-bit float with 1 sign, 4 exponent and 3 mantissa bits, exponent bias
7, subnormals, no infinities, NaN = S.1111.111), each tensor with one fp32
descale factor; the value a code stands for is ``descale * decode(code)``.
The attention of those values is the plain definition (``attention_ref``).

``decode_e4m3`` writes the format definition out; it shares nothing with the
CUDA path.
"""

from __future__ import annotations

import numpy as np

from .attention import attention_ref


def decode_e4m3(codes) -> np.ndarray:
    """Exact float64 values of E4M3 codes (uint8): sign * 2^(e-7) * (1 + m/8)
    for exponent field e in 1..15, sign * 2^-6 * (m/8) for e = 0, and NaN for
    the all-ones exponent and mantissa (the format has no infinities)."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((b & 0x80) != 0, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    subnormal = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, subnormal, normal)
    val = np.where((e == 15) & ((b & 0x7) == 7), np.nan, val)
    return sign * val


def attention_fp8_ref(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float, scale: float,
                      causal: bool = False, kv_lens=None):
    """Exact attention of FP8 inputs: ``q8 [B,H,Sq,D]``, ``k8``/``v8
    [B,H,Sk,D]`` E4M3 codes (uint8), per-tensor descales (taken as the fp32
    values a kernel receives, widened).  Returns ``attention_ref`` of the
    decoded, descaled tensors: ``(O float64, LSE float64)``."""
    qd, kd, vd = (float(np.float32(x)) for x in (q_descale, k_descale, v_descale))
    return attention_ref(decode_e4m3(q8) * qd, decode_e4m3(k8) * kd, decode_e4m3(v8) * vd, scale,
                         causal=causal, kv_lens=kv_lens)
