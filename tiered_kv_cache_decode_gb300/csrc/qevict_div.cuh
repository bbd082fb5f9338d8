// Division of the quantiser without a correctly rounded division per element.
#pragma once
#include <cuda_runtime.h>

namespace qevict {

// The correctly rounded fp32 quotient a / b, given rb = RN(1 / b): the product
// a * rb is within about an ulp of the quotient, the FMA gives its residual
// a - q0 * b exactly, and one more FMA with the reciprocal corrects q0 to the
// rounded quotient. This is the final correction step of P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990 (division through a reciprocal
// and fused multiply-adds). The step assumes no underflow: where the quotient
// is subnormal (|a| < 2^-126 b) the result can differ from the rounded
// quotient in its last bits, but both round to the integer 0, so the codes
// the quantiser derives agree. The quantiser calls it with b a positive finite
// fp16 scale and quotients of at most a few hundred; tests/test_gpu_division.py
// checks both properties over every positive finite fp16 divisor.
__device__ __forceinline__ float div_by_recip(float a, float b, float rb) {
    const float q0 = __fmul_rn(a, rb);
    const float r = __fmaf_rn(-q0, b, a);
    return __fmaf_rn(r, rb, q0);
}

}  // namespace qevict
