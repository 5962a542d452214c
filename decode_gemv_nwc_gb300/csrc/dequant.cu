// dequant.cu -- fp8 e4m3 rows to BF16 weights for prefill.
//
// "Qwen3-4B-NWC-fp8" (model card): weight-only e4m3 with a symmetric per-output-channel scale;
// prefill dequantizes the weights to BF16 and calls cuBLAS. Element (n, k) becomes the BF16
// nearest (ties to even) to the FP32 product e4m3(q[n, k]) * s_n; a NaN code gives 0x7FC0.
// The e4m3 bytes come from nwc_decode of an fp8 blob (bit-exact), so prefill runs the
// library's decoder, this kernel, then a BF16 GEMM.
//
// Memory-bound elementwise pass (N K bytes read, 2 N K written): each thread takes 8
// consecutive columns of one row, with one 8-byte load and one 16-byte store when the rows
// keep that alignment, else element by element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nwc.h"

namespace {

// Two e4m3 codes (low byte first) widened exactly to FP32 through the hardware e4m3x2 -> f16x2
// conversion (subnormals included; S.1111.111 becomes a NaN).
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
    float lo, hi;
    asm("{\n\t.reg .b16 c, l, u;\n\t.reg .b32 h;\n\t"
        "cvt.u16.u32 c, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, c;\n\t"
        "mov.b32 {l, u}, h;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, u;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(two & 0xFFFFu));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint32_t bf16_bits(float p) {
    return isnan(p) ? 0x7FC0u : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(p));
}

__global__ void dequant_fp8_kernel(const uint8_t *__restrict__ q, int64_t ld_q, const float *__restrict__ scales,
                                   int64_t n, int64_t k, uint16_t *__restrict__ out, int64_t ld_out, bool vec) {
    const int64_t chunks = (k + 7) / 8;
    const int64_t total = n * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / chunks, c0 = (i - r * chunks) * 8;
        const float s = scales[r];
        const uint8_t *qr = q + r * ld_q + c0;
        uint16_t *orow = out + r * ld_out + c0;
        if (vec && c0 + 8 <= k) {
            const uint2 b = *reinterpret_cast<const uint2 *>(qr);
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint32_t two = ((j < 2 ? b.x : b.y) >> (16 * (j & 1))) & 0xFFFFu;
                const float2 v = e4m3x2_to_f32(two);
                w[j] = bf16_bits(v.x * s) | bf16_bits(v.y * s) << 16;
            }
            *reinterpret_cast<uint4 *>(orow) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            for (int j = 0; j < 8 && c0 + j < k; j++) {
                const float v = e4m3x2_to_f32(qr[j]).x;
                orow[j] = (uint16_t)bf16_bits(v * s);
            }
        }
    }
}

}  // namespace

extern "C" nwc_status nwc_dequantize_fp8(const uint8_t *q, int64_t ld_q, const float *scales, int64_t n, int64_t k,
                                         uint16_t *out, int64_t ld_out, nwc_stream stream) {
    if (n < 0 || k < 0 || ld_q < k || ld_out < k) return NWC_ERR_INVALID_ARG;
    if (n == 0 || k == 0) return NWC_OK;
    if (!q || !scales || !out) return NWC_ERR_INVALID_ARG;
    const bool vec = (reinterpret_cast<uintptr_t>(q) % 8) == 0 && ld_q % 8 == 0 &&
                     (reinterpret_cast<uintptr_t>(out) % 16) == 0 && ld_out % 8 == 0;
    const int64_t work = n * ((k + 7) / 8);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return NWC_ERR_CUDA;
    const int threads = 256;
    const int64_t want = (work + threads - 1) / threads, cap = (int64_t)sms * 8;
    const int grid = (int)(want < cap ? want : cap);
    dequant_fp8_kernel<<<grid, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, ld_q, scales, n, k, out,
                                                                                    ld_out, vec);
    return cudaGetLastError() == cudaSuccess ? NWC_OK : NWC_ERR_CUDA;
}
