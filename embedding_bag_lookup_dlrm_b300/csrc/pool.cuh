// pool.cuh -- the pooling add of a bf16 table row into fp32 sums, shared by
// the lookup kernels.
#pragma once

#include <stdint.h>

namespace dlrm {

// lo += low bf16 half of w, hi += high half.  add.f32.bf16 converts the bf16
// operand to fp32 exactly and rounds the sum once: the same result as an fp32
// add of the widened value, in one instruction per element.
__device__ __forceinline__ void add_bf16_pair(float& lo, float& hi, uint32_t w)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w));
}

}  // namespace dlrm
