// tq2_quant.h -- launcher of the ternary producer (tq2_quant.cu).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace tq2 {
// f32 weights [N][K] (device) -> BlockTQ2_0_g128 AoS blocks (device), N*(K/128)*34 bytes.
cudaError_t launch_quantize(const float* w, uint8_t* aos, int64_t N, int64_t K, cudaStream_t st);
}  // namespace tq2
