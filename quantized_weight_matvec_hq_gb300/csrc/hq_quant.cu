// hq_quant.cu -- the data-preparation step on the GPU: fp32 weights to Q8_0,
// Q4_0 and per-output-channel int8.
//
// Formats: "One Native Stack for Private, Continuously-Learning AI", section
// "The Unified Quant Core" (Q8_0 = fp16 d + 32 int8 in 34 B, Q4_0 = fp16 d +
// 16 bytes of nibbles in 18 B, ggml's layouts).  Int8: "Blue -- porting
// zen-nano (Qwen3-0.6B) to deterministic on-chain inference", section
// "Quantization recipe (validated)" (s_w[o] = max|W[o,:]|/127, round(W/s_w)).
//
// Q4_K: the same page's section "Ported Versus Novel" (every format taken
// verbatim from ggml): a super-block of 256 weights in 144 B = fp16 d, fp16
// dmin, 12 B of six-bit sub-block scales and mins, 128 B of nibbles; encoded
// with a plain min/max reading (the pages give no encoder).
//
// Every decision that turns a float into an integer code is taken in IEEE
// fp32 with correctly rounded division (no fast-math), so the bytes are the
// same on any conforming implementation of the same reading.
#include <cuda_fp16.h>
#include <math.h>

#include "hq_internal.h"

namespace hq {

// One thread per 32-weight block.
__global__ void __launch_bounds__(256)
quantize_q8_0_kernel(const float *__restrict__ W, uint8_t *__restrict__ out, long long n_blocks) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    const float4 *src = reinterpret_cast<const float4 *>(W + b * 32);
    float w[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = src[i];
        w[4 * i] = t.x; w[4 * i + 1] = t.y; w[4 * i + 2] = t.z; w[4 * i + 3] = t.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w[j]));
    const float d = __fdiv_rn(amax, 127.0f);
    // a block is 2-byte aligned: store it as 17 halfwords (d, then quant pairs)
    unsigned short *blk = reinterpret_cast<unsigned short *>(out + b * 34);
    blk[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        int q0 = 0, q1 = 0;
        if (d != 0.f) {
            q0 = max(-127, min(127, (int)roundf(__fdiv_rn(w[j], d))));
            q1 = max(-127, min(127, (int)roundf(__fdiv_rn(w[j + 1], d))));
        }
        blk[1 + j / 2] = (unsigned short)((q0 & 0xff) | ((q1 & 0xff) << 8));
    }
}

__global__ void __launch_bounds__(256)
quantize_q4_0_kernel(const float *__restrict__ W, uint8_t *__restrict__ out, long long n_blocks) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    const float4 *src = reinterpret_cast<const float4 *>(W + b * 32);
    float w[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = src[i];
        w[4 * i] = t.x; w[4 * i + 1] = t.y; w[4 * i + 2] = t.z; w[4 * i + 3] = t.w;
    }
    // the signed element of largest magnitude, first one on ties
    float amax = 0.f, m = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float a = fabsf(w[j]);
        if (a > amax) { amax = a; m = w[j]; }
    }
    const float d = __fdiv_rn(m, -8.0f);
    unsigned short *blk = reinterpret_cast<unsigned short *>(out + b * 18);
    blk[0] = __half_as_ushort(__float2half_rn(d));
    int n[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        n[j] = 8;
        if (d != 0.f) n[j] = max(0, min(15, (int)floorf(__fadd_rn(__fdiv_rn(w[j], d), 8.5f))));
    }
    // byte j = element j (low nibble) | element j+16 (high nibble); two bytes per store
#pragma unroll
    for (int j = 0; j < 16; j += 2)
        blk[1 + j / 2] = (unsigned short)((n[j] | (n[j + 16] << 4)) | ((n[j + 1] | (n[j + 17] << 4)) << 8));
}

// One thread per Q4_K super-block.  Per 32-weight sub-block j: mn = min(0,
// min w), mx = max w, scale_j = (mx - mn)/15, min_j = -mn; d = (largest
// scale)/63 and dmin = (largest min)/63 stored fp16; sc_j = round(scale_j *
// 63/largest scale), m_j likewise, both at most 63; then with a = d sc_j and b
// = dmin m_j from the stored fp16 values, q = round((w + b)/a) clamped to
// [0, 15] (0 when a is 0).  Packing: bytes 4..15 carry the six-bit fields (see
// the header), bytes 16..143 hold four groups of 32 bytes, sub-block 2g in the
// low nibbles of group g and sub-block 2g+1 in the high nibbles.
__global__ void __launch_bounds__(128)
quantize_q4_k_kernel(const float *__restrict__ W, uint8_t *__restrict__ out, long long n_sb) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_sb) return;
    const float *w = W + b * 256;
    float scale[8], minv[8], max_scale = 0.f, max_min = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float mn = w[32 * j], mx = w[32 * j];
        for (int l = 1; l < 32; ++l) {
            const float v = w[32 * j + l];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        if (mn > 0.f) mn = 0.f;
        scale[j] = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        minv[j] = -mn;
        if (scale[j] > max_scale) max_scale = scale[j];
        if (minv[j] > max_min) max_min = minv[j];
    }
    const unsigned short dh = __half_as_ushort(__float2half_rn(__fdiv_rn(max_scale, 63.0f)));
    const unsigned short mh = __half_as_ushort(__float2half_rn(__fdiv_rn(max_min, 63.0f)));
    const float inv_s = max_scale > 0.f ? __fdiv_rn(63.0f, max_scale) : 0.f;
    const float inv_m = max_min > 0.f ? __fdiv_rn(63.0f, max_min) : 0.f;
    int sc[8], mq[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sc[j] = max(0, min(63, (int)roundf(__fmul_rn(scale[j], inv_s))));
        mq[j] = max(0, min(63, (int)roundf(__fmul_rn(minv[j], inv_m))));
    }
    uint32_t s12[3] = {0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s12[0] |= (uint32_t)(sc[j] | ((sc[j + 4] >> 4) << 6)) << (8 * j);
        s12[1] |= (uint32_t)(mq[j] | ((mq[j + 4] >> 4) << 6)) << (8 * j);
        s12[2] |= (uint32_t)((sc[j + 4] & 15) | ((mq[j + 4] & 15) << 4)) << (8 * j);
    }
    uint4 *blk = reinterpret_cast<uint4 *>(out + b * 144);     // 144 = 9 x 16 B
    blk[0] = make_uint4((uint32_t)dh | ((uint32_t)mh << 16), s12[0], s12[1], s12[2]);
    const float dq = __half2float(__ushort_as_half(dh)), mqf = __half2float(__ushort_as_half(mh));
    uint32_t *qs = reinterpret_cast<uint32_t *>(out + b * 144 + 16);
    for (int g = 0; g < 4; ++g) {
        const float a0 = __fmul_rn(dq, (float)sc[2 * g]), b0 = __fmul_rn(mqf, (float)mq[2 * g]);
        const float a1 = __fmul_rn(dq, (float)sc[2 * g + 1]), b1 = __fmul_rn(mqf, (float)mq[2 * g + 1]);
        for (int l = 0; l < 32; l += 4) {
            uint32_t word = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int lo = 0, hi = 0;
                if (a0 > 0.f) lo = max(0, min(15, (int)roundf(__fdiv_rn(__fadd_rn(w[64 * g + l + i], b0), a0))));
                if (a1 > 0.f) hi = max(0, min(15, (int)roundf(__fdiv_rn(__fadd_rn(w[64 * g + 32 + l + i], b1), a1))));
                word |= (uint32_t)(lo | (hi << 4)) << (8 * i);
            }
            qs[8 * g + l / 4] = word;
        }
    }
}

// One CTA per row: scale = max|w|/127, q = round(w/scale) in [-127, 127].
__global__ void __launch_bounds__(256)
quantize_i8_rows_kernel(const float *__restrict__ W, int8_t *__restrict__ Wq, float *__restrict__ scale,
                        long long cols) {
    const long long row = blockIdx.x;
    const float *w = W + row * cols;
    float amax = 0.f;
    for (long long j = threadIdx.x; j < cols; j += blockDim.x) amax = fmaxf(amax, fabsf(w[j]));
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, wmax[i]);
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) scale[row] = s;
    for (long long j = threadIdx.x; j < cols; j += blockDim.x) {
        int q = 0;
        if (s != 0.f) q = max(-127, min(127, (int)roundf(__fdiv_rn(w[j], s))));
        Wq[row * cols + j] = (int8_t)q;
    }
}

hq_status launch_quantize(int fmt, const float *W, void *out, float *scale, int64_t rows,
                          int64_t cols, cudaStream_t stream) {
    if (fmt == 2) {
        note_launch();
        quantize_i8_rows_kernel<<<(unsigned)rows, 256, 0, stream>>>(W, (int8_t *)out, scale, cols);
    } else if (fmt == 3) {
        const long long nsb = rows * (cols / 256);
        note_launch();
        quantize_q4_k_kernel<<<(unsigned)((nsb + 127) / 128), 128, 0, stream>>>(W, (uint8_t *)out, nsb);
    } else {
        const long long nb = rows * (cols / 32);
        const unsigned grid = (unsigned)((nb + 255) / 256);
        note_launch();
        if (fmt == 0) quantize_q8_0_kernel<<<grid, 256, 0, stream>>>(W, (uint8_t *)out, nb);
        else quantize_q4_0_kernel<<<grid, 256, 0, stream>>>(W, (uint8_t *)out, nb);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "quantize launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}

}  // namespace hq
