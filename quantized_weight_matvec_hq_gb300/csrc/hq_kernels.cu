// hq_kernels.cu -- the quantized-weight matvec kernels for sm_103a:
// Q8_0, Q4_0 and Q4_K float matvecs, the Q8_0 MoE (expert-indexed) variant,
// and the per-output-channel int8 GEMV with gemmlowp requant.
//
// What is computed:
//  * float formats ("One Native Stack for Private, Continuously-Learning AI",
//    section "The Unified Quant Core" and the Lemma of section "The Central
//    Efficiency Thesis"): y[v][i] = sum_j d_{i,b(j)} * q_{i,j} * x[v][j] over
//    the stored blocks, fp32 accumulation, n_vec = 1..8 vectors per pass;
//  * MoE ("Economical Serving and the hanzo.ai Platform", subsection "One
//    Quant-Agnostic Core"): every routed expert through the same core;
//  * int8 ("Blue -- porting zen-nano (Qwen3-0.6B) to deterministic on-chain
//    inference", section "Quantization recipe (validated)"): int32 sum of
//    int8 products, then SaturatingRoundingDoublingHighMul and
//    RoundingDivideByPOT per output channel, saturated to int8.
//
// GB300 design (the pages' lane-strided HIP kernel is prior art only):
//  * HBM-bound: each weight byte is read once per call.  A producer warp
//    stages weights into shared memory with 2-D TMA tensor copies (one per
//    stage of 32*R rows x one K chunk), completing on mbarriers, with
//    evict-first L2 hints; consumer warps never load weights from global.
//  * Lane l of a consumer warp owns output rows l, l+32, ... of the tile: a
//    row's partial sum never crosses lanes, and all lanes read the same x
//    element at once, so x comes from shared memory as broadcasts and is
//    reused across the R rows a lane holds.
//  * Bank-conflict-free row reads: a 256-column chunk of a row is 272 B
//    (Q8_0) or 144 B (Q4_0), an odd number of 16-byte units, so 8 lanes
//    reading 16-byte units of 8 consecutive rows hit 8 distinct bank groups;
//    int8 chunks are 128 B with the TMA 128-byte swizzle.
//  * int8 / nibble -> fp32 without conversion instructions: the byte goes
//    into the mantissa of 2^23 (prmt), and 2^23 + bias is subtracted exactly
//    with a packed fp32x2 add; products are packed fp32x2 FMAs.  The block sum
//    is scaled by the block's fp16 d once per block -- or, at two or more
//    vectors, d is folded into each weight by one exact packed fma (q d is
//    formed before it multiplies x), which frees the per-block sums'
//    registers for a second row per lane.
//  * Column-split stages: all consumer warps work on every stage, each on its
//    own blocks, decoded at a run-time offset so that one copy of the
//    unrolled decode serves every warp.
//  * Matrices with few row tiles split K over a thread-block cluster; the
//    partial sums are combined through distributed shared memory in a fixed
//    order (no atomics, so results are deterministic).  Large matrices run
//    persistent CTAs over row tiles.
//  * Every wait is bounded (hq_device.cuh); nothing traps.
#include <cudaTypedefs.h>
#include <limits.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "hq_device.cuh"
#include "hq_internal.h"

#ifndef HQ_PART
#define HQ_PART 0
#endif
#if HQ_PART == 1
#define HQ_PART_NAME(f) f##_q4_0
#elif HQ_PART == 4
#define HQ_PART_NAME(f) f##_q4_k
#else
#define HQ_PART_NAME(f) f##_q8_0
#endif

namespace hq {

constexpr int kMaxPairs = 256;      // MoE: n_vec * n_active

// ------------------------------------------------------------------ format policies
// Each policy states the block geometry, the TMA box of one K chunk of one
// row, the accumulator type, and the per-chunk decode + multiply-add.

constexpr uint32_t kMagic = 0x4B000000u;                    // fp32 2^23

__device__ __forceinline__ float byte_as_float(uint32_t word, int byte) {
    // 2^23 + value of byte `byte` of `word`: the byte lands in the low mantissa bits
    return __uint_as_float(prmt(word, kMagic, 0x7540u | (uint32_t)byte));
}

struct PolQ8_0 {
    static constexpr int kBlockBytes = 34;
    static constexpr int kChunkCols = 256;          // 8 blocks
    static constexpr int kChunkBytes = 272;         // per row, = 17 x 16 B
    static constexpr int kBoxInner = 68;            // uint32 words per chunk row
    static constexpr int kXElemBytes = 4;           // fp32 activations
    static constexpr int kUnits = 8;                // blocks per chunk, split across consumer warps
    static constexpr bool kSwizzle = false;
    static constexpr int kConsWarps = 2;            // memory-bound: few warps per CTA, more CTAs
    static constexpr int kConsWarpsFewAcc = 2;
    static constexpr bool kComputeBound = false;
    static constexpr bool kColSplit = false;        // see PolColSplit
    static constexpr bool kRuntimeCols = false;     // column-split decode at a run-time offset (consume_pair)
    static constexpr bool kNibbles = false;         // 4-bit quants (decode-bound launch policies)
    using Acc = float2;
    using Red = float;

    // Per lane: R rows x blocks [B0, B0+NB) of one chunk of the stage.  The
    // quant byte q XOR 0x80 (= q + 128, in [1, 255]) is placed by one prmt in
    // the low mantissa bits of 2^23, and a packed add of -(2^23 + 128) leaves
    // q exactly: every product q * x is then formed exactly inside the FMA and
    // the running sums only ever hold partial sums of q * x, so the rounding is
    // bounded by the sizes of |q * x|, whatever the signs and magnitudes of x.
    template <int NV, int R, int B0, int NB>
    __device__ __forceinline__ static void consume(const uint8_t *__restrict__ wt,
                                                   const uint8_t *__restrict__ xt8, int lane,
                                                   Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8);
        constexpr int NCH = (R * NV >= 4) ? 1 : 2;               // independent FMA chains
        const float2 kOff = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
        const uint4 *rowp[R];
        uint4 c0[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            rowp[r] = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes);
            c0[r] = rowp[r][2 * B0];
        }
#pragma unroll
        for (int b = B0; b < B0 + NB; ++b) {
            // window = 16-byte units 2b..2b+2 of the row chunk; block b starts at its byte 2b
            uint32_t win[R][12];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 c1 = rowp[r][2 * b + 1], c2 = rowp[r][2 * b + 2];
                win[r][0] = c0[r].x; win[r][1] = c0[r].y; win[r][2] = c0[r].z; win[r][3] = c0[r].w;
                win[r][4] = c1.x; win[r][5] = c1.y; win[r][6] = c1.z; win[r][7] = c1.w;
                win[r][8] = c2.x; win[r][9] = c2.y; win[r][10] = c2.z; win[r][11] = c2.w;
                c0[r] = c2;
            }
            float2 s[R][NV][NCH];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int c = 0; c < NCH; ++c) s[r][v][c] = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 32 * b + 4 * g);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float f[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int o = 2 * b + 2 + 4 * g + i;      // window byte of quant 4g+i
                        f[i] = byte_as_float(win[r][o >> 2] ^ 0x80808080u, o & 3);
                    }
                    const float2 q01 = fadd2(make_float2(f[0], f[1]), kOff);
                    const float2 q23 = fadd2(make_float2(f[2], f[3]), kOff);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        float2 &sv = s[r][v][g % NCH];
                        sv = ffma2(q01, make_float2(xv[v].x, xv[v].y), sv);
                        sv = ffma2(q23, make_float2(xv[v].z, xv[v].w), sv);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t sw = win[r][b >> 1];               // fp16 d at window byte 2b
                const unsigned short hb = (b & 1) ? (unsigned short)(sw >> 16) : (unsigned short)(sw & 0xffffu);
                const float d = __half2float(__ushort_as_half(hb));
                const float2 dd = make_float2(d, d);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float2 t = s[r][v][0];
                    if (NCH == 2) t = fadd2(t, s[r][v][NCH - 1]);
                    acc[r][v] = ffma2(dd, t, acc[r][v]);
                }
            }
        }
    }
    __device__ __forceinline__ static Red finish(const Acc &a) { return a.x + a.y; }
};

// Q8_0 at one vector on short rows (at most kShortRowCols columns, twelve K
// chunks): four consumer warps share a row tile, so more of a tile's K range
// is split inside one CTA and less over a cluster of CTAs.  Measured on the
// Qwen3-0.6B-shaped token (rows of 1024 to 3072 columns): 1492 -> 1645 GB/s;
// with rows of 4096 and more columns two warps stay ahead (8B-shaped token
// 5149 against 4935 GB/s with four).
struct PolQ8_0Short : PolQ8_0 {
    static constexpr int kConsWarpsFewAcc = 4;
};
constexpr long long kShortRowCols = 3072;

// The expert-indexed kernel at one vector: three consumer warps per CTA (with a
// ring of one stage per warp, see make_plan).
struct PolQ8_0Moe : PolQ8_0 {
    static constexpr int kConsWarpsFewAcc = 3;
};

// Q8_0 at three or more vectors: the block scale is folded into each weight,
// so a lane carries several rows without per-block partial sums (their
// registers would go to the rows instead), and x, loaded once per column
// group, serves every row of the lane.  The quant byte u = q + 128 is placed
// by one prmt at bits 8..15 of 2^23: the fp32 value f = 2^23 + 256 u.  With
// d' = d / 256 one packed fma gives f d' - (2^23 + 2^15) d' = q d exactly:
// (2^23 + 2^15) d' = 257 * 2^7 * d has 9 + 11 significant bits and q d has
// 8 + 11, so both are representable and the fma's one rounding of its exact
// result is none.  The running sums then hold partial sums of w x only.
__device__ __forceinline__ float byte_mid_as_float(uint32_t word, int byte) {
    // 2^23 + 256 * (byte `byte` of `word`)
    return __uint_as_float(prmt(word, kMagic, 0x7604u | ((uint32_t)byte << 4)));
}

struct PolQ8_0Wide : PolQ8_0 {
    static constexpr int kConsWarps = 4;            // column split: each warp two blocks of every stage
    static constexpr int kConsWarpsFewAcc = 4;
    static constexpr bool kComputeBound = true;     // the FP32 pipe, not HBM, sets the pace at eight vectors
    static constexpr bool kRuntimeCols = true;      // see consume_pair

    // block 2p + H of the chunk: words 8H .. 8H + 8 of the pair at byte 68p
    // (block 0: d in word 0's low half, quant bytes 2..33; block 1: d in word
    // 8's high half, quant bytes in words 9..16)
    template <int NV, int R, int H>
    __device__ __forceinline__ static void consume_half(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8) + 64 * p + 32 * H;
        uint32_t w[R][9];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t *rp =
                reinterpret_cast<const uint32_t *>(wt + (lane + 32 * r) * kChunkBytes + 68 * p) + 8 * H;
#pragma unroll
            for (int k = 0; k < 9; ++k) w[r][k] = rp[k] ^ 0x80808080u;
        }
        float2 dd[R], cc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned short hb = (unsigned short)((H ? (w[r][0] >> 16) : (w[r][0] & 0xffffu)) ^ 0x8080u);
            const float dq = __half2float(__ushort_as_half(hb)) * 0.00390625f;
            const float c = -8421376.0f * dq;
            dd[r] = make_float2(dq, dq);
            cc[r] = make_float2(c, c);
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            float4 xv[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v)
                xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 4 * g);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float f[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int o = 2 * H + 2 + 4 * g + i;          // byte of quant 4g+i from word 8H
                    f[i] = byte_mid_as_float(w[r][o >> 2], o & 3);
                }
                const float2 w01 = ffma2(make_float2(f[0], f[1]), dd[r], cc[r]);
                const float2 w23 = ffma2(make_float2(f[2], f[3]), dd[r], cc[r]);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    acc[r][v] = ffma2(w01, make_float2(xv[v].x, xv[v].y), acc[r][v]);
                    acc[r][v] = ffma2(w23, make_float2(xv[v].z, xv[v].w), acc[r][v]);
                }
            }
        }
    }
    // Blocks 2p and 2p + 1 of the stage's chunk for R rows per lane.  The pair
    // is 68 bytes from byte 68p of each row chunk: 17 words from a 4-byte
    // aligned start, the same word and byte positions for every p.  So p is a
    // run-time value and one copy of this code serves all four warps of a
    // column split (four copies with constant offsets overflow the SM's
    // instruction cache at these unroll depths).
    template <int NV, int R>
    __device__ __forceinline__ static void consume_pair(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        consume_half<NV, R, 0>(wt, xt8, lane, p, acc);
        consume_half<NV, R, 1>(wt, xt8, lane, p, acc);
    }
};

// Q8_0 at three or more vectors on launches that split K over clusters: eight
// consumer warps, each one block of every stage, so that the launch's few CTAs
// (1.7 per SM on the 8B-shaped o, q|k|v and down) bring twice the warps.
struct PolQ8_0Wide8 : PolQ8_0Wide {
    static constexpr int kConsWarps = 8;
    static constexpr int kConsWarpsFewAcc = 8;

    template <int NV, int R>
    __device__ __forceinline__ static void consume_one(const uint8_t *__restrict__ wt,
                                                       const uint8_t *__restrict__ xt8, int lane, int b,
                                                       Acc (&acc)[R][NV]) {
        if (b & 1) consume_half<NV, R, 1>(wt, xt8, lane, b >> 1, acc);
        else consume_half<NV, R, 0>(wt, xt8, lane, b >> 1, acc);
    }
};

// Q4_0 nibble decode, one and-or per element: a nibble at bit p in {0, 4, 8,
// 12}, masked in place and ORed into the exponent of 2^23, is the fp32 value
// 2^23 + n * 2^p (exact: the mantissa has 23 bits); adding -(2^23 + 8 * 2^p)
// leaves (n - 8) * 2^p exactly, so the running sums only ever hold partial
// sums of signed weight times x.  The exponent bits live in a register the
// compiler cannot see through, so the mask-and-OR stays one lop3 with the
// mask as its immediate.
__device__ __forceinline__ uint32_t opaque_magic() {
    uint32_t m;
    asm volatile("mov.b32 %0, 0x4B000000;" : "=r"(m));
    return m;
}
template <uint32_t MASK>
__device__ __forceinline__ float nib(uint32_t w, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "n"(MASK), "r"(magic));   // (w & MASK) | magic
    return __uint_as_float(r);
}

// Two adjacent quant bytes always lie in one 16-bit half of a word (the
// upper half is shifted down once), so every pair of low nibbles sits at bits
// (0, 8) and every pair of high nibbles at bits (4, 12); the two positions of
// a pair are summed apart and their 2^p factors are removed once per block by
// exact powers of two.
struct PolQ4_0 {
    static constexpr int kBlockBytes = 18;
    static constexpr int kChunkCols = 256;          // 8 blocks
    static constexpr int kChunkBytes = 144;         // per row, = 9 x 16 B
    static constexpr int kBoxInner = 36;            // uint32 words per chunk row
    static constexpr int kXElemBytes = 4;
    static constexpr int kUnits = 8;
    static constexpr bool kSwizzle = false;
    static constexpr int kConsWarps = 4;            // nibble decode is ALU-heavy: more warps hide its latency
    static constexpr int kConsWarpsFewAcc = 4;      // n_vec 1 (two rows per lane; see make_plan's ring)
    static constexpr bool kComputeBound = true;     // decode, not HBM, sets the pace
    static constexpr bool kColSplit = false;
    static constexpr bool kRuntimeCols = false;     // column-split decode at a run-time offset (consume_pair)
    static constexpr bool kNibbles = true;
    using Acc = float2;
    using Red = float;

    // per lane: R rows x blocks [B0, B0+NB) of one chunk of the stage
    template <int NV, int R, int B0, int NB>
    __device__ __forceinline__ static void consume(const uint8_t *__restrict__ wt,
                                                   const uint8_t *__restrict__ xt8, int lane,
                                                   Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8);
        const float2 kBiasLo = make_float2(-8388616.0f, -8390656.0f);   // -(2^23 + 8), -(2^23 + 8 * 2^8)
        const float2 kBiasHi = make_float2(-8388736.0f, -8421376.0f);   // -(2^23 + 8 * 2^4), -(2^23 + 8 * 2^12)
        const float2 kSixteenth = make_float2(0.0625f, 0.0625f);
        const uint32_t magic = opaque_magic();
        const uint4 *rowp[R];
        uint4 c0[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            rowp[r] = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes);
            c0[r] = rowp[r][B0];
        }
#pragma unroll
        for (int b = B0; b < B0 + NB; ++b) {
            uint32_t win[R][8], sw[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 c1 = rowp[r][b + 1];
                win[r][0] = c0[r].x; win[r][1] = c0[r].y; win[r][2] = c0[r].z; win[r][3] = c0[r].w;
                win[r][4] = c1.x; win[r][5] = c1.y; win[r][6] = c1.z; win[r][7] = c1.w;
                sw[r] = win[r][b >> 1];
                c0[r] = c1;
            }
            float2 slo[R][NV], shi[R][NV];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v) slo[r][v] = shi[r][v] = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 32 * b + 4 * g);
                const bool high = g >= 4;
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int t = (4 * g + 2 * h) & 15;
                        const int o = 2 * b + 2 + t;
                        const uint32_t w = (o & 2) ? (win[r][o >> 2] >> 16) : win[r][o >> 2];
                        const float2 q = high
                            ? fadd2(make_float2(nib<0xF0u>(w, magic), nib<0xF000u>(w, magic)), kBiasHi)
                            : fadd2(make_float2(nib<0xFu>(w, magic), nib<0xF00u>(w, magic)), kBiasLo);
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            const float2 xp = h ? make_float2(xv[v].z, xv[v].w) : make_float2(xv[v].x, xv[v].y);
                            float2 &sv = high ? shi[r][v] : slo[r][v];
                            sv = ffma2(q, xp, sv);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const unsigned short hb = (b & 1) ? (unsigned short)(sw[r] >> 16) : (unsigned short)(sw[r] & 0xffffu);
                const float d = __half2float(__ushort_as_half(hb));
                const float2 dd = make_float2(d, d * 0.00390625f);          // bits 8/12 carry 2^8 more
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    acc[r][v] = ffma2(dd, ffma2(shi[r][v], kSixteenth, slo[r][v]), acc[r][v]);
            }
        }
    }
    __device__ __forceinline__ static Red finish(const Acc &a) { return a.x + a.y; }
};

// Q4_0 at one or two vectors with column-split stages: the decode of PolQ4_0
// on a pair of blocks at a run-time offset, so that one copy of it serves all
// four warps.  Blocks 2p and 2p + 1 are 36 bytes from byte 36p of each row
// chunk: 9 words from a 4-byte-aligned start, the same positions for every p.
struct PolQ4_0Pair : PolQ4_0 {
    static constexpr bool kRuntimeCols = true;

    template <int NV, int R>
    __device__ __forceinline__ static void consume_pair(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8) + 64 * p;
        const float2 kBiasLo = make_float2(-8388616.0f, -8390656.0f);   // -(2^23 + 8), -(2^23 + 8 * 2^8)
        const float2 kBiasHi = make_float2(-8388736.0f, -8421376.0f);   // -(2^23 + 8 * 2^4), -(2^23 + 8 * 2^12)
        const float2 kSixteenth = make_float2(0.0625f, 0.0625f);
        const uint32_t magic = opaque_magic();
        uint32_t w[R][9];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t *rp = reinterpret_cast<const uint32_t *>(wt + (lane + 32 * r) * kChunkBytes + 36 * p);
#pragma unroll
            for (int k = 0; k < 9; ++k) w[r][k] = rp[k];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float2 slo[R][NV], shi[R][NV];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v) slo[r][v] = shi[r][v] = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 32 * h + 4 * g);
                const bool high = g >= 4;
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = (4 * g + 2 * e) & 15;
                        const int o = 18 * h + 2 + t;              // pair byte of quant bytes t, t + 1
                        const uint32_t wd = (o & 2) ? (w[r][o >> 2] >> 16) : w[r][o >> 2];
                        const float2 q = high
                            ? fadd2(make_float2(nib<0xF0u>(wd, magic), nib<0xF000u>(wd, magic)), kBiasHi)
                            : fadd2(make_float2(nib<0xFu>(wd, magic), nib<0xF00u>(wd, magic)), kBiasLo);
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            const float2 xp = e ? make_float2(xv[v].z, xv[v].w) : make_float2(xv[v].x, xv[v].y);
                            float2 &sv = high ? shi[r][v] : slo[r][v];
                            sv = ffma2(q, xp, sv);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const unsigned short hb = h ? (unsigned short)(w[r][4] >> 16) : (unsigned short)(w[r][0] & 0xffffu);
                const float d = __half2float(__ushort_as_half(hb));
                const float2 dd = make_float2(d, d * 0.00390625f);          // bits 8/12 carry 2^8 more
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    acc[r][v] = ffma2(dd, ffma2(shi[r][v], kSixteenth, slo[r][v]), acc[r][v]);
            }
        }
    }
};

// Q4_0 at three or more vectors: as PolQ8_0Wide, two rows per lane and the
// block scale folded into each weight.  A nibble n masked in place at bit p
// and ORed into 2^23 is f = 2^23 + n 2^p; with d_p = d 2^-p one packed fma
// gives f d_p - (2^23 + 8 2^p) d_p = (n - 8) d exactly when (2^(23-p) + 8) d
// is representable, i.e. for p >= 8 inside the mantissa: p = 8, 12 and 16
// ((2^12 + 1), (2^8 + 1) and 17 times 2^3 d: 13, 9 and 5 significant bits
// times d's 11).  Of a word's four quant bytes, byte 1 lies at bits 8..15 and
// byte 2 at 16..23 as loaded; one prmt brings bytes 0 and 3 there, and two
// shifts bring the high nibbles of bytes 2 and 3 to bit 12.  Each packed pair
// then shares one p.
struct PolQ4_0Wide : PolQ4_0 {
    static constexpr bool kRuntimeCols = true;      // see consume_pair

    // block 2p + H: words 4H .. 4H + 4 of the pair at byte 36p (block 0: d in
    // word 0's low half, quant bytes 2..17; block 1: d in word 4's high half,
    // quant bytes in words 5..8)
    template <int NV, int R, int H>
    __device__ __forceinline__ static void consume_half(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8) + 64 * p + 32 * H;
        const uint32_t magic = opaque_magic();
        uint32_t w[R][5];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t *rp =
                reinterpret_cast<const uint32_t *>(wt + (lane + 32 * r) * kChunkBytes + 36 * p) + 4 * H;
#pragma unroll
            for (int k = 0; k < 5; ++k) w[r][k] = rp[k];
        }
        float2 d8[R], c8[R], d12[R], c12[R], d16[R], c16[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned short hb = H ? (unsigned short)(w[r][0] >> 16) : (unsigned short)(w[r][0] & 0xffffu);
            const float d = __half2float(__ushort_as_half(hb));
            const float e8 = d * 0.00390625f, e12 = d * 0.000244140625f, e16 = d * 0.0000152587890625f;
            d8[r] = make_float2(e8, e8);
            d12[r] = make_float2(e12, e12);
            d16[r] = make_float2(e16, e16);
            const float k8 = -8390656.0f * e8, k12 = -8421376.0f * e12, k16 = -8912896.0f * e16;
            c8[r] = make_float2(k8, k8);
            c12[r] = make_float2(k12, k12);
            c16[r] = make_float2(k16, k16);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t gw[R], gb[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                gw[r] = H ? w[r][1 + k] : __funnelshift_r(w[r][k], w[r][k + 1], 16);
                gb[r] = prmt(gw[r], 0u, 0x0300u);
            }
            {
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 4 * k);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 w01 = ffma2(make_float2(nib<0xF00u>(gb[r], magic), nib<0xF00u>(gw[r], magic)),
                                             d8[r], c8[r]);
                    const float2 w23 = ffma2(make_float2(nib<0xF0000u>(gw[r], magic), nib<0xF0000u>(gb[r], magic)),
                                             d16[r], c16[r]);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        acc[r][v] = ffma2(w01, make_float2(xv[v].x, xv[v].y), acc[r][v]);
                        acc[r][v] = ffma2(w23, make_float2(xv[v].z, xv[v].w), acc[r][v]);
                    }
                }
            }
            {
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 16 + 4 * k);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float2 w01 = ffma2(make_float2(nib<0xF000u>(gb[r], magic), nib<0xF000u>(gw[r], magic)),
                                             d12[r], c12[r]);
                    const float2 w23 = ffma2(make_float2(nib<0xF000u>(gw[r] >> 8, magic),
                                                         nib<0xF000u>(gw[r] >> 16, magic)),
                                             d12[r], c12[r]);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        acc[r][v] = ffma2(w01, make_float2(xv[v].x, xv[v].y), acc[r][v]);
                        acc[r][v] = ffma2(w23, make_float2(xv[v].z, xv[v].w), acc[r][v]);
                    }
                }
            }
        }
    }
    // Blocks 2p and 2p + 1 of the stage's chunk: 36 bytes from byte 36p of each
    // row chunk, 9 words from a 4-byte-aligned start, the same positions for
    // every p, so p is a run-time value.
    template <int NV, int R>
    __device__ __forceinline__ static void consume_pair(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        consume_half<NV, R, 0>(wt, xt8, lane, p, acc);
        consume_half<NV, R, 1>(wt, xt8, lane, p, acc);
    }
};

// Q4_0 at three to five vectors on K-split launches: eight consumer warps,
// each one block of every stage (as PolQ8_0Wide8), with PolQ4_0Wide's decode.
struct PolQ4_0Wide8 : PolQ4_0Wide {
    static constexpr int kConsWarps = 8;
    static constexpr int kConsWarpsFewAcc = 8;

    template <int NV, int R>
    __device__ __forceinline__ static void consume_one(const uint8_t *__restrict__ wt,
                                                       const uint8_t *__restrict__ xt8, int lane, int b,
                                                       Acc (&acc)[R][NV]) {
        if (b & 1) consume_half<NV, R, 1>(wt, xt8, lane, b >> 1, acc);
        else consume_half<NV, R, 0>(wt, xt8, lane, b >> 1, acc);
    }
};

// Q4_K ("One Native Stack ...", sections "The Unified Quant Core" and "Ported
// Versus Novel": ggml's super-block of 256 weights in 144 B).  A 256-column
// chunk of a row is exactly one super-block: 16-byte unit 0 holds fp16 d,
// fp16 dmin and the 12 bytes of six-bit sub-block scales sc_j and mins m_j;
// units 1..8 hold four groups of 32 quant bytes, sub-block 2g in the low
// nibbles of group g and sub-block 2g+1 in the high nibbles; the weight is
// w = d sc_j q - dmin m_j.
//
// Every weight is formed in fp32 before it multiplies x: the nibble is placed
// in the mantissa of 2^23 (one lop3) and 2^23 removed exactly, leaving q 2^p;
// then one packed fma gives (d sc_j 2^-p) (q 2^p) - dmin m_j = w, rounded once.
// So the running sums hold partial sums of w x, and the rounding is bounded by
// the products |w x| themselves, as for the symmetric formats.
struct PolQ4_K {
    static constexpr int kBlockBytes = 18;          // bytes per 32 columns (a super-block: 144 B per 256)
    static constexpr int kChunkCols = 256;          // one super-block per row chunk
    static constexpr int kChunkBytes = 144;         // = 9 x 16 B
    static constexpr int kBoxInner = 36;            // uint32 words per chunk row
    static constexpr int kXElemBytes = 4;
    static constexpr int kUnits = 8;                // sub-blocks per chunk
    static constexpr bool kSwizzle = false;
    static constexpr int kConsWarps = 4;
    static constexpr int kConsWarpsFewAcc = 4;
    static constexpr bool kComputeBound = true;
    static constexpr bool kColSplit = false;
    static constexpr bool kRuntimeCols = false;     // column-split decode at a run-time offset (consume_pair)
    static constexpr bool kNibbles = true;
    using Acc = float2;
    using Red = float;

    // six-bit scale (sel 0) or min (sel 1) of sub-block J from the header words
    // s0 = bytes 4..7, s1 = bytes 8..11, s2 = bytes 12..15 of the super-block
    template <int J, int SEL>
    __device__ __forceinline__ static uint32_t six(uint32_t s0, uint32_t s1, uint32_t s2) {
        if constexpr (J < 4) return ((SEL ? s1 : s0) >> (8 * J)) & 63u;
        else {
            const uint32_t lo4 = (s2 >> (8 * (J - 4) + 4 * SEL)) & 15u;
            const uint32_t hi2 = ((SEL ? s1 : s0) >> (8 * (J - 4) + 6)) & 3u;
            return lo4 | (hi2 << 4);
        }
    }

    // sub-blocks [B0, B0 + 2): quant group B0 / 2 of every row the lane holds
    template <int NV, int R, int B0, int NB>
    __device__ __forceinline__ static void consume(const uint8_t *__restrict__ wt,
                                                   const uint8_t *__restrict__ xt8, int lane,
                                                   Acc (&acc)[R][NV]) {
        static_assert(NB == 2 && B0 % 2 == 0, "one quant group per call");
        constexpr int G = B0 / 2;
        const float *xt = reinterpret_cast<const float *>(xt8);
        const float2 kM = make_float2(-8388608.0f, -8388608.0f);          // -2^23
        const uint32_t magic = opaque_magic();
        float2 alo[R], ahi[R], blo[R], bhi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4 hdr = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[0];
            const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
            const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
            const float a0 = d * (float)six<B0, 0>(hdr.y, hdr.z, hdr.w);
            const float a1 = d * (float)six<B0 + 1, 0>(hdr.y, hdr.z, hdr.w);
            const float b0 = dm * (float)six<B0, 1>(hdr.y, hdr.z, hdr.w);
            const float b1 = dm * (float)six<B0 + 1, 1>(hdr.y, hdr.z, hdr.w);
            alo[r] = make_float2(a0, a0 * 0.00390625f);                  // nibbles at bits 0 and 8
            ahi[r] = make_float2(a1 * 0.0625f, a1 * 0.000244140625f);     // nibbles at bits 4 and 12
            blo[r] = make_float2(-b0, -b0);
            bhi[r] = make_float2(-b1, -b1);
        }
        float2 shi[R][NV];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) shi[r][v] = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 2; ++u) {                   // the group's two 16-byte units
            uint32_t qw[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 q = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[1 + 2 * G + u];
                qw[r][0] = q.x; qw[r][1] = q.y; qw[r][2] = q.z; qw[r][3] = q.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {            // quant bytes 4k .. 4k+3 of the group
                const int k = 4 * u + kk;
                float4 xl[NV], xh[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    xl[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 64 * G + 4 * k);
                    xh[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 64 * G + 32 + 4 * k);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t w = h ? (qw[r][kk] >> 16) : qw[r][kk];
                        const float2 qlo = fadd2(make_float2(nib<0xFu>(w, magic), nib<0xF00u>(w, magic)), kM);
                        const float2 qhi = fadd2(make_float2(nib<0xF0u>(w, magic), nib<0xF000u>(w, magic)), kM);
                        const float2 wlo = ffma2(alo[r], qlo, blo[r]);
                        const float2 whi = ffma2(ahi[r], qhi, bhi[r]);
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            const float2 xpl = h ? make_float2(xl[v].z, xl[v].w) : make_float2(xl[v].x, xl[v].y);
                            const float2 xph = h ? make_float2(xh[v].z, xh[v].w) : make_float2(xh[v].x, xh[v].y);
                            acc[r][v] = ffma2(wlo, xpl, acc[r][v]);
                            shi[r][v] = ffma2(whi, xph, shi[r][v]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) acc[r][v] = fadd2(acc[r][v], shi[r][v]);
    }
    __device__ __forceinline__ static Red finish(const Acc &a) { return a.x + a.y; }
};

// Q4_K with column-split stages (one vector, and four or more at two rows per
// lane): one copy of the decode for all four warps: warp p takes quant group p
// (sub-blocks 2p and 2p + 1) with p in a register, and reads the two
// sub-blocks' six-bit scales and mins with run-time shifts.  The weights are
// formed as in PolQ4_K.
struct PolQ4_KWide : PolQ4_K {
    static constexpr bool kRuntimeCols = true;      // see consume_pair

    __device__ __forceinline__ static uint32_t six_rt(int j, int sel, uint32_t s0, uint32_t s1, uint32_t s2) {
        const uint32_t sm = sel ? s1 : s0;
        if (j < 4) return (sm >> (8 * j)) & 63u;
        const uint32_t lo4 = (s2 >> (8 * (j - 4) + 4 * sel)) & 15u;
        const uint32_t hi2 = (sm >> (8 * (j - 4) + 6)) & 3u;
        return lo4 | (hi2 << 4);
    }

    template <int NV, int R>
    __device__ __forceinline__ static void consume_pair(const uint8_t *__restrict__ wt,
                                                        const uint8_t *__restrict__ xt8, int lane, int p,
                                                        Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8) + 64 * p;
        const float2 kM = make_float2(-8388608.0f, -8388608.0f);          // -2^23
        const uint32_t magic = opaque_magic();
        float2 alo[R], ahi[R], blo[R], bhi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4 hdr = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[0];
            const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
            const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
            const float a0 = d * (float)six_rt(2 * p, 0, hdr.y, hdr.z, hdr.w);
            const float a1 = d * (float)six_rt(2 * p + 1, 0, hdr.y, hdr.z, hdr.w);
            const float b0 = dm * (float)six_rt(2 * p, 1, hdr.y, hdr.z, hdr.w);
            const float b1 = dm * (float)six_rt(2 * p + 1, 1, hdr.y, hdr.z, hdr.w);
            alo[r] = make_float2(a0, a0 * 0.00390625f);                  // nibbles at bits 0 and 8
            ahi[r] = make_float2(a1 * 0.0625f, a1 * 0.000244140625f);     // nibbles at bits 4 and 12
            blo[r] = make_float2(-b0, -b0);
            bhi[r] = make_float2(-b1, -b1);
        }
        // with few accumulators the second sub-block's products go to a second set
        // (two independent FMA chains per output)
        constexpr bool kTwo = NV * R <= 2;
        float2 acc2[R][NV];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) acc2[r][v] = make_float2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 2; ++u) {                   // the group's two 16-byte units
            uint32_t qw[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 q = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[1 + 2 * p + u];
                qw[r][0] = q.x; qw[r][1] = q.y; qw[r][2] = q.z; qw[r][3] = q.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {            // quant bytes 4k .. 4k+3 of the group
                const int k = 4 * u + kk;
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {        // sub-block 2p (low nibbles), then 2p + 1
                    float4 xv[NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 32 * hi + 4 * k);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t w = h ? (qw[r][kk] >> 16) : qw[r][kk];
                            const float2 q = hi ? fadd2(make_float2(nib<0xF0u>(w, magic), nib<0xF000u>(w, magic)), kM)
                                                : fadd2(make_float2(nib<0xFu>(w, magic), nib<0xF00u>(w, magic)), kM);
                            const float2 wq = hi ? ffma2(ahi[r], q, bhi[r]) : ffma2(alo[r], q, blo[r]);
#pragma unroll
                            for (int v = 0; v < NV; ++v) {
                                const float2 xp = h ? make_float2(xv[v].z, xv[v].w) : make_float2(xv[v].x, xv[v].y);
                                float2 &av = (kTwo && hi) ? acc2[r][v] : acc[r][v];
                                av = ffma2(wq, xp, av);
                            }
                        }
                    }
                }
            }
        }
        if constexpr (kTwo) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v) acc[r][v] = fadd2(acc[r][v], acc2[r][v]);
        }
    }
};

// Q4_K at three and four vectors on K-split launches: eight consumer warps,
// warp b one sub-block of every stage (the low nibbles of quant group b / 2
// for even b, the high nibbles for odd b), as PolQ8_0Wide8 does for Q8_0.
struct PolQ4_KWide8 : PolQ4_KWide {
    static constexpr int kConsWarps = 8;
    static constexpr int kConsWarpsFewAcc = 8;

    template <int NV, int R, int HI>
    __device__ __forceinline__ static void consume_sub(const uint8_t *__restrict__ wt,
                                                       const uint8_t *__restrict__ xt8, int lane, int p,
                                                       Acc (&acc)[R][NV]) {
        const float *xt = reinterpret_cast<const float *>(xt8) + 64 * p + 32 * HI;
        const float2 kM = make_float2(-8388608.0f, -8388608.0f);          // -2^23
        const uint32_t magic = opaque_magic();
        float2 aa[R], bb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4 hdr = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[0];
            const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xffffu)));
            const float dm = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
            const float a = d * (float)six_rt(2 * p + HI, 0, hdr.y, hdr.z, hdr.w);
            const float b = dm * (float)six_rt(2 * p + HI, 1, hdr.y, hdr.z, hdr.w);
            aa[r] = HI ? make_float2(a * 0.0625f, a * 0.000244140625f)      // nibbles at bits 4 and 12
                       : make_float2(a, a * 0.00390625f);                  // nibbles at bits 0 and 8
            bb[r] = make_float2(-b, -b);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            uint32_t qw[R][4];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint4 q = reinterpret_cast<const uint4 *>(wt + (lane + 32 * r) * kChunkBytes)[1 + 2 * p + u];
                qw[r][0] = q.x; qw[r][1] = q.y; qw[r][2] = q.z; qw[r][3] = q.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = 4 * u + kk;
                float4 xv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    xv[v] = *reinterpret_cast<const float4 *>(xt + v * kChunkCols + 4 * k);
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t w = h ? (qw[r][kk] >> 16) : qw[r][kk];
                        const float2 q = HI ? fadd2(make_float2(nib<0xF0u>(w, magic), nib<0xF000u>(w, magic)), kM)
                                            : fadd2(make_float2(nib<0xFu>(w, magic), nib<0xF00u>(w, magic)), kM);
                        const float2 wq = ffma2(aa[r], q, bb[r]);
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            const float2 xp = h ? make_float2(xv[v].z, xv[v].w) : make_float2(xv[v].x, xv[v].y);
                            acc[r][v] = ffma2(wq, xp, acc[r][v]);
                        }
                    }
                }
            }
        }
    }
    template <int NV, int R>
    __device__ __forceinline__ static void consume_one(const uint8_t *__restrict__ wt,
                                                       const uint8_t *__restrict__ xt8, int lane, int b,
                                                       Acc (&acc)[R][NV]) {
        if (b & 1) consume_sub<NV, R, 1>(wt, xt8, lane, b >> 1, acc);
        else consume_sub<NV, R, 0>(wt, xt8, lane, b >> 1, acc);
    }
};

struct PolI8 {
    static constexpr int kChunkCols = 128;          // one 128-byte swizzle span
    static constexpr int kChunkBytes = 128;
    static constexpr int kBoxInner = 128;           // uint8 elements per chunk row
    static constexpr int kXElemBytes = 1;
    static constexpr int kUnits = 8;                // 16-byte units per chunk
    static constexpr bool kSwizzle = true;
    static constexpr int kConsWarps = 2;
    static constexpr int kConsWarpsFewAcc = 2;
    static constexpr bool kComputeBound = false;
    static constexpr bool kColSplit = false;
    static constexpr bool kRuntimeCols = false;     // column-split decode at a run-time offset (consume_pair)
    static constexpr bool kNibbles = false;
    using Acc = int;
    using Red = int;

    template <int NV, int R, int U0, int NU>
    __device__ __forceinline__ static void consume(const uint8_t *__restrict__ wt,
                                                   const uint8_t *__restrict__ xt, int lane,
                                                   Acc (&acc)[R][NV]) {
#pragma unroll
        for (int u = U0; u < U0 + NU; ++u) {
            int4 xu[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) xu[v] = *reinterpret_cast<const int4 *>(xt + v * kChunkCols + 16 * u);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = lane + 32 * r;
                // 128-byte swizzle: 16-byte unit u of tile row `row` sits at unit u ^ (row & 7)
                const int4 w = *reinterpret_cast<const int4 *>(wt + row * kChunkBytes + 16 * (u ^ (row & 7)));
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    acc[r][v] = __dp4a(w.x, xu[v].x, acc[r][v]);
                    acc[r][v] = __dp4a(w.y, xu[v].y, acc[r][v]);
                    acc[r][v] = __dp4a(w.z, xu[v].z, acc[r][v]);
                    acc[r][v] = __dp4a(w.w, xu[v].w, acc[r][v]);
                }
            }
        }
    }
    __device__ __forceinline__ static Red finish(const Acc &a) { return a; }
};

// Column-split stages (the 4-bit formats at one vector, whose decode sets the
// pace; Q8_0 at three or more vectors and the 4-bit formats at four or more,
// where the FP32 pipe does).  Every consumer warp consumes
// every stage, each its own blocks of all the stage's rows; the tile's partial
// sums are added across the warps at its end.  The stage's x tile is loaded
// once for all warps.  A stage is then in use for a
// quarter of the time one warp would need for it, so the same shared memory
// keeps more bytes in flight.
template <class Base>
struct PolColSplit : Base {
    static constexpr bool kColSplit = true;
};

template <class Acc> __device__ __forceinline__ Acc zero_acc();
template <> __device__ __forceinline__ float2 zero_acc<float2>() { return make_float2(0.f, 0.f); }
template <> __device__ __forceinline__ int zero_acc<int>() { return 0; }

// gemmlowp requant, restated: SRDHM(a, m) = floor((a*m + 2^30) / 2^31) except
// a = m = INT32_MIN -> INT32_MAX; RDivByPOT(v, e) = v / 2^e rounded to nearest,
// ties away from zero; then saturate to int8.
__device__ __forceinline__ int requant_i8(int acc, int mult, int shift) {
    long long v;
    if (acc == INT_MIN && mult == INT_MIN) v = INT_MAX;
    else v = ((long long)acc * (long long)mult + (1LL << 30)) >> 31;   // arithmetic shift = floor
    const int e = min(max(shift, 0), 31);
    if (e > 0) {
        const long long mag = v < 0 ? -v : v;
        const long long q = (mag + (1LL << (e - 1))) >> e;
        v = v < 0 ? -q : q;
    }
    return (int)min(max(v, -128LL), 127LL);
}

// ------------------------------------------------------------------ kernel arguments / layout

constexpr int kMaxSplit = 8;        // CTAs per cluster when K is split

struct KArgs {
    CUtensorMap tmW;          // weights: {inner units per row, total rows}
    CUtensorMap tmX;          // dense x: {cols, n_vec}
    void *y;                  // fp32 [n_vec][rows] / MoE [n_vec][n_active][rows] / int8 [n_vec][rows]
    const float *x;           // MoE: x base, gathered per vector with bulk copies
    const int32_t *ids;       // MoE: expert ids [n_vec][n_active]
    const int32_t *mult;      // int8: [rows]
    const int32_t *shift;     // int8: [rows]
    uint32_t *fault;
    long long rows;           // rows of one matrix
    long long cols;
    long long n_experts;
    int n_chunks;             // cols / kChunkCols
    int num_tiles;            // row tiles of one matrix
    int stages;               // depth of the CTA's stage ring
    int ksplit;               // CTAs per cluster along K (1: persistent over tiles)
    int n_vec;
    int n_active;
    int x_per_slot;
    const uint16_t *lora_B;   // QLoRA epilogue (lora_rank > 0): bf16 [rows][lora_rank]
    const float *lora_u;      //   u = A x, fp32 [n_vec][lora_rank]
    float lora_scale;         //   y += lora_scale * B u
    int lora_rank;
    int moe_epi;              // MoE epilogue: kEpiNone, kEpiSwiglu or kEpiCombine
    const float *router_w;    //   combine: router weights [n_vec][n_active]
    int gsplit;               // combine: CTAs per row tile (a cluster when > 1), over the tile's expert groups
    int lay_ks;               // gather-buffer slots in the shared-memory layout
    int ids_ready;            // MoE: the expert ids were written before the previous kernel in the stream
};

// MoE epilogues.  SwiGLU: an expert's gate and up rows are interleaved (row 2i
// gate i, row 2i+1 up i) and y receives h_i = silu(gate_i) * up_i, [n_vec][n_active][rows/2].
// Combine: y [n_vec][rows] receives the router-weighted sum over each token's
// slots.  A cluster of G <= kCombineCluster CTAs owns one row tile (G is as
// large as one wave of CTAs allows); CTA r takes the expert groups r, r + G,
// ... and keeps its weighted per-token partial sums in shared memory; the
// leader adds the CTAs' partials in rank order through distributed shared
// memory.  No atomics, no workspace, and a fixed summation order.
constexpr int kEpiNone = 0, kEpiSwiglu = 1, kEpiCombine = 2;
constexpr int kCombineCluster = 8;

// Consumer warps per CTA for a format and accumulator count.
template <class P, int NV, int R>
__host__ __device__ constexpr int cons_warps() { return (NV * R <= 2) ? P::kConsWarpsFewAcc : P::kConsWarps; }

template <class P, int NV, int R, bool MOE>
struct Layout {
    static constexpr int TR = 32 * R;                                   // rows per tile
    static constexpr int WT = TR * P::kChunkBytes;                      // weight tile bytes
    static constexpr int kAlign = P::kSwizzle ? 1024 : 128;            // TMA destination alignment
    static constexpr int XT = ((NV * P::kChunkCols * P::kXElemBytes + kAlign - 1) / kAlign) * kAlign;
    static constexpr int ST = WT + XT;                                  // stage bytes
    static_assert(WT % kAlign == 0 && ST % kAlign == 0, "stage alignment");
    static constexpr size_t kMiscBytes = 16 + (MOE ? 5 * kMaxPairs * 4 : 0);   // abort flag, MoE tables
    // s = ring stages, ks = CTAs per cluster along K (the gather buffer exists only when ks > 1)
    __host__ __device__ static size_t red_off(int s) { return (size_t)s * ST; }
    __host__ __device__ static size_t part_off(int s) {
        return red_off(s) + (size_t)cons_warps<P, NV, R>() * TR * NV * 4;
    }
    __host__ __device__ static size_t bar_off(int s, int ks) {
        return part_off(s) + (ks > 1 ? (size_t)ks * TR * NV * 4 : 0);
    }
    __host__ __device__ static size_t misc_off(int s, int ks) { return bar_off(s, ks) + (size_t)(2 * s + 2) * 8; }
    __host__ __device__ static size_t total(int s, int ks) { return misc_off(s, ks) + kMiscBytes + kAlign; }
};

// MoE groups: (token, slot) pairs sorted by expert, cut into groups of at most
// NV pairs sharing one expert; group g covers sorted[gstart[g] .. + gsize[g]).
struct MoeTables {
    int *sorted, *gstart, *gsize, *gexpert, *n_groups, *ids;    // ids: the call's expert ids, staged
};

// The QLoRA term scale * sum_k B[row][k] * u[v][k] of one output (bf16 B,
// its bits the upper half of an fp32).
__device__ __forceinline__ float lora_term(const uint16_t *B, const float *u, float scale, int rank,
                                           int v, long long row) {
    const uint16_t *b = B + row * rank;
    const float *uv = u + (long long)v * rank;
    float t = 0.f;
    for (int k = 0; k < rank; ++k) t = fmaf(__uint_as_float((uint32_t)b[k] << 16), uv[k], t);
    return scale * t;
}

template <class P, bool MOE>
__device__ __forceinline__ void store_out(const KArgs &a, const MoeTables &mt, int g, int v,
                                          long long row, typename P::Red val) {
    if constexpr (std::is_same<typename P::Red, int>::value) {
        reinterpret_cast<int8_t *>(a.y)[(long long)v * a.rows + row] =
            (int8_t)requant_i8(val, a.mult[row], a.shift[row]);
    } else {
        const long long p = MOE ? (long long)mt.sorted[mt.gstart[g] + v] : (long long)v;
        if (!MOE && a.lora_rank > 0) val += lora_term(a.lora_B, a.lora_u, a.lora_scale, a.lora_rank, v, row);
        reinterpret_cast<float *>(a.y)[p * a.rows + row] = val;
    }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Entry e of this CTA's own combine partial sums (kept in the gather buffer).
template <class T>
__device__ __forceinline__ float csum_own(const T *part, int e) { return reinterpret_cast<const float *>(part)[e]; }

// SwiGLU epilogue of one MoE tile: sums[v * TR + rr] holds the tile's reduced
// outputs for the group's vector v; rows rr (even) and rr + 1 are a gate/up
// pair, and h goes to y[pair (token, slot)][tile * TR/2 + rr/2].
__device__ __forceinline__ void store_swiglu_tile(const KArgs &a, const MoeTables &mt, int g, int tile, int TR,
                                                  int m, const float *sums, int tid, int nthr) {
    const long long half = a.rows / 2;
    for (int e = tid; e < (TR / 2) * m; e += nthr) {
        const int v = e / (TR / 2), pr = e % (TR / 2);
        const long long i = (long long)tile * (TR / 2) + pr;
        if (i >= half) continue;
        const long long p = mt.sorted[mt.gstart[g] + v];
        const float gate = sums[v * TR + 2 * pr], up = sums[v * TR + 2 * pr + 1];
        reinterpret_cast<float *>(a.y)[p * half + i] = silu_f(gate) * up;
    }
}

// A whole chunk for one warp, in pieces of two units; the empty asm between
// pieces keeps the compiler from hoisting every piece's shared loads at once
// (which would cost registers and occupancy, not latency).
template <class P, int NV, int R>
__device__ __forceinline__ void consume_chunk(const uint8_t *wt, const uint8_t *xt, int lane,
                                              typename P::Acc (&acc)[R][NV]) {
    P::template consume<NV, R, 0, 2>(wt, xt, lane, acc);
    asm volatile("" ::: "memory");
    P::template consume<NV, R, 2, 2>(wt, xt, lane, acc);
    asm volatile("" ::: "memory");
    P::template consume<NV, R, 4, 2>(wt, xt, lane, acc);
    asm volatile("" ::: "memory");
    P::template consume<NV, R, 6, 2>(wt, xt, lane, acc);
}

// Column split: warp w of four consumes blocks (units) 2w and 2w + 1 of every
// stage, with w a run-time value (one copy of the decode for all four warps).
template <class P, int NV, int R>
__device__ __forceinline__ void consume_cols(const uint8_t *wt, const uint8_t *xt, int lane, int warp,
                                             typename P::Acc (&acc)[R][NV]) {
    constexpr int CW = cons_warps<P, NV, R>();
    static_assert((CW == 4 || CW == 8) && P::kUnits == 8 && P::kRuntimeCols,
                  "four warps of two units each (or eight of one), decoded at a run-time offset");
    if constexpr (CW == 8) P::template consume_one<NV, R>(wt, xt, lane, warp, acc);
    else P::template consume_pair<NV, R>(wt, xt, lane, warp, acc);
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ the kernel
//
// CTA = CW consumer warps (cons_warps<P,NV,R>) + 1 producer warp, several
// CTAs per SM (each with its own producer: one thread issuing copies cannot
// keep HBM busy for a whole SM).  The producer walks the CTA's work items
// (row tiles, or (expert group, row tile) for MoE) and fills one stage of the
// CTA's ring per K chunk.  Fill n (chunk j of a tile, counted over the CTA's
// items) lands in stage n mod S and is consumed whole by warp n mod CW, which
// owns the tile's 32*R rows (R per lane); S is a multiple of CW, so every
// stage has one owner.  A tile ends with a fixed-order reduction over the CW
// warps; with a K split, the CTAs of a cluster then combine their partials
// through DSMEM.  With column-split stages (PolColSplit) every warp consumes
// every fill (its own blocks of the tile's rows), and the stage is freed by
// all CW warps.
//
// Programmatic dependent launch: the kernel lets the next one in the stream
// start as soon as it is resident, issues the weight copies of its first
// stages at once (weights are never written by another kernel), and waits for
// the previous kernel only before it touches x, expert ids or y.

// CTAs per SM the kernel is compiled for (its register cap follows): more
// when a lane holds few accumulators, fewer when it holds many or the CTA has
// four or more consumer warps.
template <class P, int NV, int R>
constexpr int ctas_per_sm() {
    // Q8_0 at three or more vectors: 75-104 registers, three CTAs of four consumer warps
    if constexpr (std::is_base_of<PolQ8_0Wide8, P>::value || std::is_base_of<PolQ4_0Wide8, P>::value ||
                  std::is_base_of<PolQ4_KWide8, P>::value)
        return 2;
    if constexpr (std::is_base_of<PolQ8_0Wide, P>::value || std::is_base_of<PolQ4_0Wide, P>::value ||
                  std::is_base_of<PolQ4_KWide, P>::value)
        return 3;
    // Q4_0 at 2-6 vectors: its 96-116 registers leave room for a third CTA
    // (8B-shaped token n_vec 3 / 4: 1865 / 1606 -> 1939 / 1651 GB/s; n_vec 2,
    // with a ring of one stage per warp: 2520 -> 2733 GB/s)
    // (Q4_K: up to 5; at 6 vectors its weights-then-products decode needs more)
    if constexpr (P::kNibbles) if (NV >= 2 && NV <= (std::is_same<P, PolQ4_K>::value ? 5 : 6)) return 3;
    return cons_warps<P, NV, R>() >= 8 ? 2
         : cons_warps<P, NV, R>() >= 4 ? ((NV * R <= 2) ? 3 : 2)
                                        : ((NV * R <= 2) ? 5 : 3);
}

template <class P, int NV, int R, bool MOE>
__global__ void __launch_bounds__(32 * (cons_warps<P, NV, R>() + 1), ctas_per_sm<P, NV, R>())
matvec_tma_kernel(const __grid_constant__ KArgs a) {
    using L = Layout<P, NV, R, MOE>;
    using Acc = typename P::Acc;
    using Red = typename P::Red;
    constexpr int TR = L::TR, WT = L::WT, ST = L::ST;
    constexpr int XV = P::kChunkCols * P::kXElemBytes;                  // x bytes per vector per chunk
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // align by offsetting the __shared__ array itself (not through an integer
    // cast), so the compiler keeps every access in the shared address space
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + L::kAlign - 1) & ~uint32_t(L::kAlign - 1)) - raw);
    const int S = a.stages;
    Red *red = reinterpret_cast<Red *>(smem + L::red_off(S));
    Red *part = reinterpret_cast<Red *>(smem + L::part_off(S));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off(S, a.lay_ks));
    uint64_t *empty = full + S;
    uint64_t *gather_bar = empty + S;           // K split: the leader CTA counts the others' partials
    int *misc = reinterpret_cast<int *>(smem + L::misc_off(S, a.lay_ks));
    volatile int *abort_flag = misc;
    const MoeTables mt{misc + 4, misc + 4 + kMaxPairs, misc + 4 + 2 * kMaxPairs,
                       misc + 4 + 3 * kMaxPairs, misc + 1, misc + 4 + 4 * kMaxPairs};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nthreads = blockDim.x;
    constexpr int CW = cons_warps<P, NV, R>();      // S % CW == 0 unless columns are split (see make_plan)
    constexpr bool SH = P::kColSplit;               // every warp consumes every stage

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(&full[i]), 1);
            mbar_init(smem_u32(&empty[i]), SH ? CW : 1);   // column split: every warp frees the stage
        }
        mbar_init(smem_u32(gather_bar), (uint32_t)max(a.ksplit - 1, 1));
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_launch_dependents();
    if constexpr (MOE) {
        // ids may come from the previous kernel (a router): wait for it first,
        // unless the caller vouches that they were written before it
        if (!a.ids_ready) griddep_wait();
        // Group the (token, slot) pairs by expert; every CTA derives the same
        // table.  The ids are read from global memory once, in parallel, and
        // every later look-up is a shared-memory read.
        const int P_ = a.n_vec * a.n_active;
        for (int p = threadIdx.x; p < P_; p += nthreads) mt.ids[p] = a.ids[p];
        __syncthreads();
        for (int p = threadIdx.x; p < P_; p += nthreads) {
            const int e = mt.ids[p];
            const long long ke = (e >= 0 && e < a.n_experts) ? e : a.n_experts;
            int rank = 0;
            for (int q = 0; q < P_; ++q) {
                const int eq = mt.ids[q];
                const long long kq = (eq >= 0 && eq < a.n_experts) ? eq : a.n_experts;
                rank += (kq < ke) || (kq == ke && q < p);
            }
            mt.sorted[rank] = p;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int ng = 0, bad = 0;
            for (int i = 0; i < P_;) {
                const int e = mt.ids[mt.sorted[i]];
                if (e < 0 || e >= a.n_experts) { bad = 1; ++i; continue; }
                int j = i + 1;
                while (j < P_ && j - i < NV && mt.ids[mt.sorted[j]] == e) ++j;
                mt.gstart[ng] = i; mt.gsize[ng] = j - i; mt.gexpert[ng] = e; ++ng;
                i = j;
            }
            *mt.n_groups = ng;
            misc[2] = bad;
            if (bad && blockIdx.x == 0) atomicOr(a.fault, kFaultExpertId);
        }
        __syncthreads();
        if (blockIdx.x == 0 && misc[2]) {          // outputs of invalid ids become NaN
            if (a.ids_ready) griddep_wait();       // y may still be in use by the previous kernel
            const long long out_rows = a.moe_epi == kEpiSwiglu ? a.rows / 2 : a.rows;
            for (int p = 0; p < P_ && a.moe_epi != kEpiCombine; ++p) {   // combine: the leader writes NaN sums
                const int e = mt.ids[p];
                if (e >= 0 && e < a.n_experts) continue;
                for (long long r = threadIdx.x; r < out_rows; r += nthreads)
                    reinterpret_cast<float *>(a.y)[(long long)p * out_rows + r] = __int_as_float(0x7fc00000);
            }
        }
    }
    __syncthreads();

    const int n_work = MOE ? (*mt.n_groups) * a.num_tiles : a.num_tiles;
    const bool split = a.ksplit > 1;
    const bool gs = MOE && a.moe_epi == kEpiCombine;   // combine: gsplit CTAs split a row tile's groups
    // every CTA of the cluster has initialised its barriers before any remote access
    if (split) cluster_arrive_relaxed();
    const int rank = (split || (gs && a.gsplit > 1)) ? (int)cluster_ctarank() : 0;
    // split: one tile per cluster; gs: groups rank, rank + gsplit, ... of the cluster's tile
    const int work0 = split ? (int)(blockIdx.x / a.ksplit)
                            : gs ? rank * a.num_tiles + (int)(blockIdx.x / a.gsplit) : (int)blockIdx.x;
    const int wstep = split ? max(n_work, 1) : gs ? a.gsplit * a.num_tiles : (int)gridDim.x;
    const int k0 = split ? (int)((long long)rank * a.n_chunks / a.ksplit) : 0;
    const int k1 = split ? (int)((long long)(rank + 1) * a.n_chunks / a.ksplit) : a.n_chunks;
    const int nloc = k1 - k0;

    if (warp == CW) {
        // ---------------- producer: one elected lane issues every copy
        if (lane == 0) {
            const uint64_t polW = l2_evict_first_policy();
            const uint64_t polX = l2_evict_last_policy();
            prefetch_tensormap(&a.tmW);
            if (!MOE) prefetch_tensormap(&a.tmX);
            // The weights never depend on the previous kernel: the first S stages'
            // weight tiles are requested at once, and only then does the producer
            // wait for the previous kernel (x and the expert ids may come from it).
            uint32_t n_pre = 0;
            if (!MOE || a.ids_ready) {
                for (int work = work0; work < n_work && n_pre < (uint32_t)S; work += wstep) {
                    long long row0 = (long long)(work % a.num_tiles) * TR;
                    int m = NV;
                    if (MOE) {
                        const int g = work / a.num_tiles;
                        m = mt.gsize[g];
                        row0 += (long long)mt.gexpert[g] * a.rows;
                    }
                    for (int j = 0; j < nloc && n_pre < (uint32_t)S; ++j, ++n_pre) {
                        const uint32_t fb = smem_u32(&full[n_pre]);
                        mbar_arrive_expect_tx(fb, WT + m * XV);
                        tma_load_2d(smem_u32(smem + (size_t)n_pre * ST), &a.tmW, (k0 + j) * P::kBoxInner,
                                    (int)row0, fb, polW);
                    }
                }
                griddep_wait();
            }
            uint32_t n = 0;
            for (int work = work0; work < n_work; work += wstep) {
                const int tile = work % a.num_tiles;
                int m = NV, g = 0;
                long long row0 = (long long)tile * TR;
                if (MOE) {
                    g = work / a.num_tiles;
                    m = mt.gsize[g];
                    row0 += (long long)mt.gexpert[g] * a.rows;
                }
                for (int j = 0; j < nloc; ++j, ++n) {
                    const int s = n % S;
                    uint8_t *st = smem + (size_t)s * ST;
                    const uint32_t fb = smem_u32(&full[s]);
                    const int kc = k0 + j;
                    if (n >= n_pre) {
                        if (n >= (uint32_t)S) mbar_wait(smem_u32(&empty[s]), ((n / S) - 1) & 1, abort_flag, a.fault);
                        mbar_arrive_expect_tx(fb, WT + m * XV);
                        tma_load_2d(smem_u32(st), &a.tmW, kc * P::kBoxInner, (int)row0, fb, polW);
                    }
                    if (!MOE) {
                        tma_load_2d(smem_u32(st + WT), &a.tmX, kc * P::kChunkCols, 0, fb, polX);
                    } else {
                        for (int i = 0; i < m; ++i) {
                            const int p = mt.sorted[mt.gstart[g] + i];
                            const long long xr = a.x_per_slot ? p : p / a.n_active;
                            bulk_load(smem_u32(st + WT + i * XV),
                                      a.x + xr * a.cols + (long long)kc * P::kChunkCols, XV, fb, polX);
                        }
                    }
                }
            }
            // no copy may still be landing in shared memory when the CTA exits
            for (int s = 0; s < S; ++s) {
                if (n <= (uint32_t)s) continue;
                const uint32_t last = n - 1 - ((n - 1 - s) % S);             // last fill of stage s
                const uint32_t bar = smem_u32(&full[s]);
                const long long t0 = sm_cycles();
                while (!mbar_try_wait(bar, (last / S) & 1))
                    if (sm_cycles() - t0 > kWaitTimeoutCycles) break;
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers
        if (split) cluster_wait();               // the leader's gather buffer and barrier exist
        float *csum = reinterpret_cast<float *>(part);   // gs: weighted partial sums [n_vec][TR]
        if (gs)
            for (int e = threadIdx.x; e < a.n_vec * TR; e += CW * 32) csum[e] = 0.f;
        griddep_wait();                          // y may still be in use by the previous kernel
        uint32_t base = 0;                       // fill number of the current item's first chunk
        for (int work = work0; work < n_work; work += wstep, base += nloc) {
            const int tile = work % a.num_tiles;
            int m = NV, g = 0;
            if (MOE) { g = work / a.num_tiles; m = mt.gsize[g]; }
            Acc acc[R][NV];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v) acc[r][v] = zero_acc<Acc>();
            // fill n lands in stage n % S and belongs to warp n % CW (S is a multiple
            // of CW): each stage is only ever consumed by one warp, in fill order,
            // so a wait can never mistake a stage's previous phase for its next.
            // Column split: every warp consumes every fill (its own blocks of the
            // stage), so each warp waits on every phase of every stage in order.
            for (int j = SH ? 0 : (warp - (int)(base % CW) + CW) % CW; j < nloc; j += SH ? 1 : CW) {
                const uint32_t n = base + j;
                const int s = n % S;
                mbar_wait(smem_u32(&full[s]), (n / S) & 1, abort_flag, a.fault);
                uint8_t *st = smem + (size_t)s * ST;
                if constexpr (!MOE) {
                    if constexpr (P::kColSplit) consume_cols<P, NV, R>(st, st + WT, lane, warp, acc);
                    else consume_chunk<P, NV, R>(st, st + WT, lane, acc);
                } else {
                    // only the group's m vectors are multiplied
                    switch (m) {
#define HQ_MOE_CASE(M_)                                                              \
    case M_:                                                                         \
        if constexpr (M_ <= NV) {                                                    \
            Acc acc_m[R][M_];                                                        \
            _Pragma("unroll") for (int r = 0; r < R; ++r)                            \
                _Pragma("unroll") for (int v = 0; v < M_; ++v) acc_m[r][v] = acc[r][v]; \
            consume_chunk<P, M_, R>(st, st + WT, lane, acc_m);                       \
            _Pragma("unroll") for (int r = 0; r < R; ++r)                            \
                _Pragma("unroll") for (int v = 0; v < M_; ++v) acc[r][v] = acc_m[r][v]; \
        }                                                                            \
        break;
                        HQ_MOE_CASE(1) HQ_MOE_CASE(2) HQ_MOE_CASE(3) HQ_MOE_CASE(4)
                        HQ_MOE_CASE(5) HQ_MOE_CASE(6) HQ_MOE_CASE(7) HQ_MOE_CASE(8)
#undef HQ_MOE_CASE
                        default: break;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            }
            // reduction of the tile over all consumer warps, in fixed warp order
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    red[(warp * NV + v) * TR + lane + 32 * r] =
                        P::finish(acc[r][v]);
            named_barrier(1, CW * 32);
            if (gs) {
                // one thread per row adds the group's members in order: two slots of a
                // token may share an expert, so a token's sum has one writer per row
                for (int rr = threadIdx.x; rr < TR; rr += CW * 32)
                    for (int v = 0; v < m; ++v) {
                        Red sum = red[v * TR + rr];
                        for (int w2 = 1; w2 < CW; ++w2) sum += red[(w2 * NV + v) * TR + rr];
                        const int p = mt.sorted[mt.gstart[g] + v];
                        float &c = csum[(p / a.n_active) * TR + rr];
                        c = fmaf(a.router_w[p], (float)sum, c);
                    }
            }
            for (int e = threadIdx.x; e < TR * m && !gs; e += CW * 32) {
                const int v = e / TR, rr = e % TR;
                Red sum = red[v * TR + rr];
                for (int w2 = 1; w2 < CW; ++w2) sum += red[(w2 * NV + v) * TR + rr];
                const long long row = (long long)tile * TR + rr;
                if (split) {
                    // this CTA's partial goes to slot `rank` of the leader's gather buffer
                    const uint32_t slot = smem_u32(&part[((size_t)rank * NV + v) * TR + rr]);
                    if constexpr (std::is_same<Red, int>::value) st_shared_cluster_s32(map_shared_rank(slot, 0), sum);
                    else st_shared_cluster_f32(map_shared_rank(slot, 0), sum);
                } else if (MOE && a.moe_epi == kEpiSwiglu) {
                    red[v * TR + rr] = sum;              // paired below (only this thread reads the slot)
                } else if (row < a.rows) {
                    store_out<P, MOE>(a, mt, g, v, row, sum);
                }
            }
            named_barrier(1, CW * 32);
            if constexpr (MOE) {
                if (!split && a.moe_epi == kEpiSwiglu) {
                    store_swiglu_tile(a, mt, g, tile, TR, m, reinterpret_cast<const float *>(red), threadIdx.x, CW * 32);
                    named_barrier(1, CW * 32);           // red is rewritten by the next item
                }
            }
            if (split && rank != 0 && threadIdx.x == 0)
                mbar_arrive_remote(map_shared_rank(smem_u32(gather_bar), 0));
        }
    }

    if (split) {
        // K was split across the cluster: the leader (rank 0) adds the ranks'
        // partials in rank order and stores the tile; the other CTAs are done.
        if (warp == CW) cluster_wait();          // the producer warp completes the cluster barrier too
        __syncthreads();                         // the leader's own partial is in `part` for all threads
        const int work = work0;
        if (rank == 0 && work < n_work) {
            if (a.ksplit > 1) mbar_wait_cluster(smem_u32(gather_bar), 0, abort_flag, a.fault);
            const int tile = work % a.num_tiles;
            int m = NV, g = 0;
            if (MOE) { g = work / a.num_tiles; m = mt.gsize[g]; }
            for (int e = threadIdx.x; e < TR * m; e += nthreads) {
                const int v = e / TR, rr = e % TR;
                Red sum = part[(size_t)v * TR + rr];
                for (int q = 1; q < a.ksplit; ++q) sum += part[((size_t)q * NV + v) * TR + rr];
                const long long row = (long long)tile * TR + rr;
                if (MOE && a.moe_epi == kEpiSwiglu) part[(size_t)v * TR + rr] = sum;    // paired below
                else if (row < a.rows) store_out<P, MOE>(a, mt, g, v, row, sum);
            }
            if constexpr (MOE) {
                if (a.moe_epi == kEpiSwiglu) {
                    __syncthreads();
                    store_swiglu_tile(a, mt, g, tile, TR, m, reinterpret_cast<const float *>(part), threadIdx.x, nthreads);
                }
            }
        }
    }

    if (gs) {
        // Every CTA of the cluster holds its weighted partial sums; the leader
        // adds them in rank order through distributed shared memory.  The second
        // cluster barrier keeps every CTA's shared memory alive until then.
        __syncwarp();
        if (a.gsplit > 1) {
            cluster_arrive_release();
            cluster_wait();
        } else {
            __syncthreads();
        }
        if (rank == 0) {
            const int tile = (int)(blockIdx.x / a.gsplit);
            const uint32_t base = smem_u32(part);
            for (int e = threadIdx.x; e < a.n_vec * TR; e += nthreads) {
                const int t = e / TR, rr = e % TR;
                const long long row = (long long)tile * TR + rr;
                if (row >= a.rows) continue;
                float pv[kCombineCluster];
#pragma unroll
                for (int q = 0; q < kCombineCluster; ++q)
                    pv[q] = q >= a.gsplit ? 0.f
                          : a.gsplit > 1 ? ld_shared_cluster_f32(map_shared_rank(base + 4u * (uint32_t)e, (uint32_t)q))
                                         : csum_own(part, e);
                float acc = pv[0];
#pragma unroll
                for (int q = 1; q < kCombineCluster; ++q) if (q < a.gsplit) acc += pv[q];
                bool valid = true;
                for (int k = 0; k < a.n_active; ++k) {
                    const int id = mt.ids[t * a.n_active + k];
                    valid &= id >= 0 && id < a.n_experts;
                }
                reinterpret_cast<float *>(a.y)[(long long)t * a.rows + row] = valid ? acc : __int_as_float(0x7fc00000);
            }
        }
        __syncwarp();
        if (a.gsplit > 1) {
            cluster_arrive_release();
            cluster_wait();
        }
    }
}

// ------------------------------------------------------------------ plain-load kernels
// Legal shapes whose rows are not 16-byte aligned (cols % 256 != 0, or int8
// cols % 128 != 0): one warp per row, lanes over blocks, small aligned loads.

template <int FMT>
__global__ void __launch_bounds__(256)
matvec_plain_kernel(const uint8_t *__restrict__ W, const float *__restrict__ x, float *__restrict__ y,
                    long long rows, long long cols, int n_vec, const uint16_t *lora_B,
                    const float *lora_u, float lora_scale, int lora_rank) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long long nb = cols / 32;
    constexpr int bb = FMT == 0 ? 34 : 18;
    float acc[8];
    for (int v = 0; v < 8; ++v) acc[v] = 0.f;
    for (long long b = lane; b < nb; b += 32) {
        const uint16_t *blk = reinterpret_cast<const uint16_t *>(W + (row * nb + b) * bb);
        const float d = __half2float(__ushort_as_half(blk[0]));
        float q[32];
#pragma unroll
        for (int h = 0; h < (bb - 2) / 2; ++h) {
            const uint32_t two = blk[1 + h];
            if (FMT == 0) {
                q[2 * h] = (float)(int8_t)(two & 0xff);
                q[2 * h + 1] = (float)(int8_t)(two >> 8);
            } else {
                q[2 * h] = (float)(int)((two & 0xf) - 8);
                q[2 * h + 16] = (float)(int)(((two >> 4) & 0xf) - 8);
                q[2 * h + 1] = (float)(int)(((two >> 8) & 0xf) - 8);
                q[2 * h + 17] = (float)(int)((two >> 12) - 8);
            }
        }
        for (int v = 0; v < n_vec; ++v) {
            const float *xv = x + (long long)v * cols + b * 32;
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) s = fmaf(q[j], xv[j], s);
            acc[v] = fmaf(d, s, acc[v]);
        }
    }
    for (int v = 0; v < n_vec; ++v) {
        float s = acc[v];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
            if (lora_rank > 0) s += lora_term(lora_B, lora_u, lora_scale, lora_rank, v, row);
            y[(long long)v * rows + row] = s;
        }
    }
}

#if HQ_PART == 2
__global__ void __launch_bounds__(256)
matvec_i8_plain_kernel(const int8_t *__restrict__ W, const int8_t *__restrict__ x,
                       const int32_t *__restrict__ mult, const int32_t *__restrict__ shift,
                       int8_t *__restrict__ y, long long rows, long long cols, int n_vec) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int *w4 = reinterpret_cast<const int *>(W + row * cols);
    for (long long j = lane; j < cols / 4; j += 32) {
        const int w = w4[j];
        for (int v = 0; v < n_vec; ++v)
            acc[v] = __dp4a(w, reinterpret_cast<const int *>(x + (long long)v * cols)[j], acc[v]);
    }
    for (int v = 0; v < n_vec; ++v) {
        int s = acc[v];
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) y[(long long)v * rows + row] = (int8_t)requant_i8(s, mult[row], shift[row]);
    }
}

__global__ void requant_debug_kernel(const int32_t *__restrict__ acc, const int32_t *__restrict__ mult,
                                     const int32_t *__restrict__ shift, int8_t *__restrict__ y,
                                     long long n, long long rows) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        y[i] = (int8_t)requant_i8(acc[i], mult[i % rows], shift[i % rows]);
}

// QLoRA down projection u[v][k] = sum_j A[k][j] * x[v][j] (A bf16 [rank][cols],
// cols % 8 == 0): one CTA of 512 threads per adapter row k, eight columns per
// thread and step, so a row of up to 4096 columns is one step and of up to
// 8192 two; then a fixed-order reduction (warp shuffles, then the 16 warps in
// order), so u is the same bit for bit on every run.  Launched as a
// programmatic dependent: it becomes resident while the previous kernel
// drains, loads its first two steps of A, and reads x (which that kernel may
// write) only after waiting for it; both steps' x loads are then in flight at
// once.  It lets the matvec that follows start at once (that kernel reads u
// only after waiting for this one).  Against one CTA of 256 threads with a
// step at a time: 8B token with rank-16 adapters 3821 -> 3937 GB/s (Q8_0),
// 2294 -> 2330 (Q4_0); 1024 threads gained more on Q4_0 (2381) but lost on
// Q8_0 (3789): a larger CTA holds more of the SM the overlapping matvec needs.
constexpr int kLoraThreads = 512;
__global__ void __launch_bounds__(kLoraThreads) lora_down_kernel(const uint16_t *__restrict__ A,
                                                                 const float *__restrict__ x,
                                                                 float *__restrict__ u, int rank, long long cols,
                                                                 int n_vec) {
    griddep_launch_dependents();
    const int k = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4 *a8 = reinterpret_cast<const uint4 *>(A + (long long)k * cols);
    const long long n8 = cols / 8;
    // A is a weight: its first two steps are read before waiting for the previous kernel
    const long long c0 = threadIdx.x, c1 = threadIdx.x + kLoraThreads;
    const uint4 w0 = c0 < n8 ? a8[c0] : make_uint4(0u, 0u, 0u, 0u);
    const uint4 w1 = c1 < n8 ? a8[c1] : make_uint4(0u, 0u, 0u, 0u);
    griddep_wait();
    float acc[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) acc[v] = 0.f;
    auto step = [&](const uint4 &w, long long c) {
        const float wf[8] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                             __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u),
                             __uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                             __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u)};
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            if (v >= n_vec) break;
            const float4 *xv = reinterpret_cast<const float4 *>(x + (long long)v * cols) + 2 * c;
            const float4 p = xv[0], q = xv[1];
            float t = acc[v];
            t = fmaf(wf[0], p.x, t); t = fmaf(wf[1], p.y, t); t = fmaf(wf[2], p.z, t); t = fmaf(wf[3], p.w, t);
            t = fmaf(wf[4], q.x, t); t = fmaf(wf[5], q.y, t); t = fmaf(wf[6], q.z, t); t = fmaf(wf[7], q.w, t);
            acc[v] = t;
        }
    };
    if (c0 < n8) step(w0, c0);
    if (c1 < n8) step(w1, c1);
    for (long long c = c1 + kLoraThreads; c < n8; c += kLoraThreads) step(a8[c], c);
    __shared__ float red[kLoraThreads / 32][8];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        float t = acc[v];
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) red[warp][v] = t;
    }
    __syncthreads();
    if (threadIdx.x < n_vec) {
        float t = 0.f;
        for (int w2 = 0; w2 < kLoraThreads / 32; ++w2) t += red[w2][threadIdx.x];
        u[(long long)threadIdx.x * rank + k] = t;
    }
}

// Test-only: a bounded wait on an mbarrier nothing arrives on (see
// hq_selftest_wait_timeout in the header).
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint32_t *fault, long long limit_cycles) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, fault, limit_cycles);
    __syncwarp();
}

#endif  // HQ_PART == 2

// ------------------------------------------------------------------ host side

namespace {

struct Plan {
    int stages = 4, ksplit = 1, grid = 1, gsplit = 1, lay_ks = 1;
    long long slots = 0;
    size_t smem = 0;
};

hq_status encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!enc) return set_error(HQ_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(HQ_ERR_LAUNCH, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return HQ_OK;
}

// Launch geometry: ctas_per_sm<P,NV,R>() CTAs per SM, the stage ring sized to
// share the SM's shared memory among them.  Row tiles are 32*R rows; when
// there are too few to fill every CTA slot, K is split across a cluster of up
// to 8 CTAs, never beyond one wave.
template <class P, int NV, int R, bool MOE>
Plan make_plan(const DeviceInfo &dev, long long n_work, int n_chunks, int regs_per_thread, int gsplit = 0) {
    using L = Layout<P, NV, R, MOE>;
    Plan p;
    const size_t budget = (size_t)dev.max_smem_optin;
    const int want = ctas_per_sm<P, NV, R>();
    constexpr int CW = cons_warps<P, NV, R>();
    // stages come in multiples of CW (one owner each), or of one when every warp
    // consumes every stage (column split)
    constexpr bool SH = P::kColSplit;
    constexpr int SQ = SH ? 1 : CW;
    // two stages per consumer warp (a double buffer each), more when room allows;
    // column split: two stages for the CTA, more when room allows
    // Q4_0 at one vector starts from one stage per warp: with four consumer
    // warps the ring then leaves room for 3 CTAs per SM (2 with two stages per
    // warp); the ring still grows below when fewer CTAs are resident.  8B-shaped
    // Q4_0 token: 3154 GB/s with three warps and two stages each, 3411 with
    // three warps and one, 3568 with four warps and one.  The MoE kernel at one
    // vector does the same with three warps (48-layer step 2399 -> 2526 GB/s),
    // and so did the dense Q8_0 kernel at two vectors before its wide policy; the dense
    // Q8_0 kernel at one vector does not (8B token 5186 -> 4607 GB/s), nor the
    // MoE kernel at four vectors (2696 -> 2579 GB/s).
    constexpr int kSpw = (((P::kNibbles || std::is_same<P, PolQ8_0Moe>::value) && NV == 1) ||
                          (P::kNibbles && NV == 2)) ? 1 : 2;
    p.stages = SH ? 2 : kSpw * SQ;
    while (L::total(p.stages + SQ, 1) * want <= budget && p.stages < 4 * SQ) p.stages += SQ;
    p.smem = L::total(p.stages, 1);
    const int regs = std::max(32, regs_per_thread);
    const long long by_regs = 65536 / (32 * (CW + 1) * ((regs + 7) / 8 * 8));
    const long long per_sm = std::max<long long>(1, std::min<long long>({by_regs, (long long)want,
                                                                          (long long)(budget / p.smem)}));
    const long long slots = (long long)dev.num_sms * per_sm;
    int ks = 1;
    p.slots = slots;
    // (the wide-vector policy's gather buffer is large: a split must leave its CTAs per SM room)
    constexpr bool kFitSplit = std::is_base_of<PolQ8_0Wide, P>::value || std::is_base_of<PolQ4_0Wide, P>::value ||
                               std::is_base_of<PolQ4_KWide, P>::value;
    while (gsplit == 0 && ks < kMaxSplit && n_work * ks * 2 <= slots && n_chunks >= 2 * ks &&
           (!kFitSplit || L::total(2, 2 * ks) * per_sm <= budget))
        ks *= 2;
    // Q4_0 (decode-bound) on launches short enough that the largest K split
    // that still fits one wave leaves each CTA at most three chunks: that split
    // fills every CTA slot (o 4096x4096: clusters of 7, 1626 -> 1880 GB/s; the
    // 8B token 2990 -> 3056).  Longer rows lost with it (down 4096x14336, 8
    // chunks per CTA: 2872 -> 2529), and so did Q4_K (token 2553 -> 2171).
    if (std::is_same<P, PolQ4_0>::value && gsplit == 0 && ks > 1 && !MOE) {
        int kf = ks;
        while (kf < kMaxSplit && n_work * (kf + 1) <= slots && n_chunks >= kf + 1) ++kf;
        if ((n_chunks + kf - 1) / kf <= 3) ks = kf;
    }
    p.ksplit = ks;
    p.gsplit = std::max(gsplit, 1);
    // gather-buffer slots: the K split's partials, or a combine's own partial sums
    const int lks = ks > 1 ? ks : (gsplit >= 1 ? 2 : 1);
    p.lay_ks = lks;
    if (gsplit >= 1) {
        p.grid = (int)n_work;                    // n_work counts the CTAs: row tiles x gsplit
    } else if (ks == 1 && P::kComputeBound) {
        // every slot filled, tiles strided over the CTAs: each SM then holds
        // about the same number of tiles, which is what a decode-bound kernel needs
        p.grid = (int)std::min<long long>(n_work, slots);
    } else if (ks == 1) {
        // the same number of tiles for every CTA: with HBM shared fairly, CTAs then finish together
        const long long per_cta = (n_work + slots - 1) / slots;
        p.grid = (int)((n_work + per_cta - 1) / per_cta);
    } else {
        p.grid = (int)(n_work * ks);
    }
    // the ring takes the shared memory the SM's resident CTAs leave: fewer CTAs
    // per SM get deeper rings, so an SM keeps about the same bytes in flight
    const long long resident = std::min<long long>(per_sm, std::max<long long>(1, (p.grid + dev.num_sms - 1) / dev.num_sms));
    int st = p.stages;
    const int st_min = SH ? 2 : CW;
    while (st > st_min && L::total(st, lks) * resident > budget) st -= SQ;    // room for the gather buffer
    while (st + SQ <= 16 && L::total(st + SQ, lks) * resident <= budget) st += SQ;
    {
        // a CTA never has more stages than fills: the shared memory it leaves
        // lets the next kernel's CTAs become resident (and start their weight
        // copies) while this one drains
        // (a group split's items are data-dependent: it keeps the full ring)
        const long long items = (ks > 1) ? 1 : gsplit >= 1 ? 1LL << 30 : (n_work + p.grid - 1) / std::max(p.grid, 1);
        const long long fills = items * ((n_chunks + ks - 1) / ks);
        const long long need = SH ? std::max<long long>(2, fills)
                                            : std::max<long long>(CW, (fills + CW - 1) / CW * CW);
        if (need < st) st = (int)need;
    }
    p.stages = st;
    p.smem = L::total(st, lks);
    return p;
}

template <class P, int NV, int R, bool MOE>
int kernel_regs() {
    static int regs = -1;
    if (regs < 0) {
        cudaFuncAttributes fa;
        regs = (cudaFuncGetAttributes(&fa, matvec_tma_kernel<P, NV, R, MOE>) == cudaSuccess) ? fa.numRegs : 128;
    }
    return regs;
}

size_t dev_smem_limit();

// Clusters of G CTAs (smem bytes each) that can be resident at once, from the
// occupancy calculator; cached per device, kernel, G and size.
template <class P, int NV, int R, bool MOE>
long long max_active_clusters(const DeviceInfo &dev, int G, size_t smem) {
    struct Entry { int device, G; size_t smem; long long n; };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;                        // launches may come from several host threads
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].device == dev.device && cache[i].G == G && cache[i].smem == smem) return cache[i].n;
    auto kern = matvec_tma_kernel<P, NV, R, MOE>;
    long long n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev_smem_limit()) == cudaSuccess &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)G, 1, 1);
        cfg.blockDim = dim3((unsigned)(32 * (cons_warps<P, NV, R>() + 1)), 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)G;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, kern, &cfg) == cudaSuccess) n = c;
    }
    cudaGetLastError();                          // a failed query only means: do not use this G
    if (used < 32) cache[used++] = Entry{dev.device, G, smem, n};
    return n;
}

size_t dev_smem_limit() {
    DeviceInfo *d = nullptr;
    return device_info(&d) == HQ_OK ? (size_t)d->max_smem_optin : 0;
}

template <class P, int NV, int R, bool MOE>
hq_status launch_tma(KArgs &a, const Plan &p, cudaStream_t stream) {
    auto kern = matvec_tma_kernel<P, NV, R, MOE>;
    // the shared-memory opt-in is raised once per device and kernel, before any
    // stream capture that launches it
    static int configured[64] = {0};
    int devi = 0;
    cudaGetDevice(&devi);
    cudaError_t e = cudaSuccess;
    if (devi < 0 || devi >= 64 || configured[devi] == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dev_smem_limit());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        // one shared-memory carveout for every launch: consecutive matvecs of
        // different sizes then never make an SM reconfigure its L1/shared split
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        if (devi >= 0 && devi < 64) configured[devi] = 1;
    }
    a.stages = p.stages;
    a.ksplit = p.ksplit;
    a.gsplit = p.gsplit;
    a.lay_ks = p.lay_ks;
    if (p.grid <= 0) return HQ_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)(32 * (cons_warps<P, NV, R>() + 1)), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.ksplit > 1 || p.gsplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)std::max(p.ksplit, p.gsplit);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e == cudaSuccess) note_launch();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "matvec launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}

// Rows per lane: two for the 4-bit formats at one or two vectors (the second
// row shares the x loads and adds independent work to a warp whose decode, not
// HBM, is the limit); one otherwise (the wide-vector policies chosen in
// with_dense_policy take two).
template <class P>
constexpr int rows_per_lane(int nv) {
    return (P::kNibbles && nv <= 2) ? 2 : 1;
}

template <class P, int NV, int R>
hq_status dense_nv_r(const DeviceInfo &dev, const void *W, const void *x, void *y, const int32_t *mult,
                     const int32_t *shift, long long rows, long long cols, const MatvecExtras *lora,
                     cudaStream_t stream) {
    constexpr bool kI8 = std::is_same<P, PolI8>::value;
    constexpr int TR = Layout<P, NV, R, false>::TR;             // rows per tile (one TMA box)
    KArgs a = {};
    long long row_bytes;
    hq_status st;
    if constexpr (kI8) {
        row_bytes = cols;
        st = encode_2d(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, (uint64_t)cols, (uint64_t)rows,
                       (uint64_t)row_bytes, P::kBoxInner, TR, true);
        if (st != HQ_OK) return st;
        st = encode_2d(&a.tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, x, (uint64_t)cols, (uint64_t)NV,
                       (uint64_t)cols, P::kChunkCols, NV, false);
    } else {
        row_bytes = cols / 32 * P::kBlockBytes;
        st = encode_2d(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, W, (uint64_t)(row_bytes / 4),
                       (uint64_t)rows, (uint64_t)row_bytes, P::kBoxInner, TR, false);
        if (st != HQ_OK) return st;
        st = encode_2d(&a.tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, (uint64_t)cols, (uint64_t)NV,
                       (uint64_t)cols * 4, P::kChunkCols, NV, false);
    }
    if (st != HQ_OK) return st;
    a.y = y;
    a.mult = mult;
    a.shift = shift;
    a.fault = dev.fault;
    a.rows = rows;
    a.cols = cols;
    a.n_chunks = (int)(cols / P::kChunkCols);
    a.num_tiles = (int)((rows + TR - 1) / TR);
    a.n_vec = NV;
    if (lora && lora->rank > 0) {
        a.lora_B = lora->B;
        a.lora_u = lora->u;
        a.lora_scale = lora->scale;
        a.lora_rank = lora->rank;
    }
    const Plan p = make_plan<P, NV, R, false>(dev, a.num_tiles, a.n_chunks, kernel_regs<P, NV, R, false>());
    return launch_tma<P, NV, R, false>(a, p, stream);
}

// The launch policy of a dense matvec: format P at NV vectors on rows of
// `cols` columns.  Calls f(policy, rows-per-lane) with the chosen policy type
// and R as an integral_constant; the launch and the test-only plan query
// (hq_debug_plan) both go through here, so they cannot disagree.
template <class P, int NV, class F>
hq_status with_dense_policy(const DeviceInfo &dev, long long rows, long long cols, F &&f) {
    constexpr int R = rows_per_lane<P>(NV);
    using RT = std::integral_constant<int, R>;
    if constexpr (std::is_same<P, PolQ8_0>::value && NV == 1) {
        // (the wide policy below lost here: 8B-shaped token 4970 -> 4581 GB/s,
        // and 4967 -> 4647 with it on the launches without a K split only,
        // although gate|up alone gained 5182 -> 5548: its four-stage ring
        // leaves the next launch no room; with three or two stages gate|up
        // itself fell to 4825 / 4056 GB/s; eight warps on the short-row K-split
        // launches alone lost too, Qwen3-0.6B token 1609 -> 1448 GB/s)
        if (cols <= kShortRowCols) return f(PolQ8_0Short{}, RT{});
        return f(P{}, RT{});
    } else if constexpr (std::is_same<P, PolQ8_0>::value) {
        // Q8_0 at two or more vectors: column-split stages of 64-row tiles, two
        // rows per lane, the scale folded into each weight (PolQ8_0Wide).  Against
        // the row-split stages of one row per lane it replaced (one 32-row share
        // of every stage per warp), the 8B-shaped token at n_vec 3 / 4 / 5 / 8:
        // 3280 / 2716 / 2045 / 1335 -> 3605 / 2952 / 2764 / 2135 GB/s; at n_vec 2,
        // against three warps each owning a stage of 32 rows, 3784 -> 4175.
        // Three rows per lane (96-row tiles) lost on the K-split launches.
        // Eight consumer warps, one block each (PolQ8_0Wide8), on launches that
        // split K and keep the same split with them (the launch's CTAs then bring
        // twice the warps): rows of at most 3072 columns at every n_vec
        // (Qwen3-0.6B-shaped token at n_vec 3 / 4 / 8: 1101 / 996 / 764 -> 1261 /
        // 1195 / 893 GB/s) and the longer rows at n_vec <= 4 (8B-shaped token at
        // n_vec 4: 2945 -> 3149; at 5 / 6 / 8 it lost 1-2 %, at 3 it tied).
        if (cols <= kShortRowCols || NV <= 4) {
            const long long tiles = (rows + 63) / 64;
            const int chunks = (int)(cols / PolQ8_0::kChunkCols);
            const Plan p4 = make_plan<PolColSplit<PolQ8_0Wide>, NV, 2, false>(dev, tiles, chunks, 0);
            const Plan p8 = make_plan<PolColSplit<PolQ8_0Wide8>, NV, 2, false>(dev, tiles, chunks, 0);
            if (p4.ksplit > 1 && p8.ksplit >= p4.ksplit)
                return f(PolColSplit<PolQ8_0Wide8>{}, std::integral_constant<int, 2>{});
        }
        return f(PolColSplit<PolQ8_0Wide>{}, std::integral_constant<int, 2>{});
    } else if constexpr (P::kNibbles && NV == 3) {
        // three vectors: one owner per stage and one row per lane, except on
        // K-split launches that keep their split with eight warps of one block
        // each (Q4_0 token 1931 -> 1959 GB/s; the four-warp wide layout lost
        // here, see below)
        const long long tiles = (rows + 63) / 64;
        const int chunks = (int)(cols / P::kChunkCols);
        if constexpr (std::is_same<P, PolQ4_0>::value) {
            const Plan p4 = make_plan<PolColSplit<PolQ4_0Wide>, NV, 2, false>(dev, tiles, chunks, 0);
            const Plan p8 = make_plan<PolColSplit<PolQ4_0Wide8>, NV, 2, false>(dev, tiles, chunks, 0);
            if (p4.ksplit > 1 && p8.ksplit >= p4.ksplit)
                return f(PolColSplit<PolQ4_0Wide8>{}, std::integral_constant<int, 2>{});
        } else {
            // (Q4_K token 1742 -> 1761 GB/s)
            const Plan p4 = make_plan<PolColSplit<PolQ4_KWide>, NV, 2, false>(dev, tiles, chunks, 0);
            const Plan p8 = make_plan<PolColSplit<PolQ4_KWide8>, NV, 2, false>(dev, tiles, chunks, 0);
            if (p4.ksplit > 1 && p8.ksplit >= p4.ksplit)
                return f(PolColSplit<PolQ4_KWide8>{}, std::integral_constant<int, 2>{});
        }
        return f(P{}, RT{});
    } else if constexpr (std::is_same<P, PolQ4_0>::value && NV >= 4) {
        // the 4-bit formats from four vectors on, where the FP32 pipe binds: as
        // Q8_0 above (Q4_0 token n_vec 4 / 6 / 8: 1658 / 1284 / 1008 -> 1681 /
        // 1326 / 1131 GB/s; at n_vec 3 it lost, 1930 -> 1730, and at 2 as well;
        // at 3 on the launches without a K split only, Q4_0 1928 -> 1852 and
        // Q4_K 1743 -> 1701).
        // Eight warps of one block each on K-split launches that keep their
        // split, as for Q8_0, at four and five vectors (token n_vec 4 1679 ->
        // 1712 GB/s); from six vectors on their 96-register bound spills.
        if constexpr (NV <= 5) {
            const long long tiles = (rows + 63) / 64;
            const int chunks = (int)(cols / PolQ4_0::kChunkCols);
            const Plan p4 = make_plan<PolColSplit<PolQ4_0Wide>, NV, 2, false>(dev, tiles, chunks, 0);
            const Plan p8 = make_plan<PolColSplit<PolQ4_0Wide8>, NV, 2, false>(dev, tiles, chunks, 0);
            if (p4.ksplit > 1 && p8.ksplit >= p4.ksplit)
                return f(PolColSplit<PolQ4_0Wide8>{}, std::integral_constant<int, 2>{});
        }
        return f(PolColSplit<PolQ4_0Wide>{}, std::integral_constant<int, 2>{});
    } else if constexpr (std::is_same<P, PolQ4_K>::value && NV >= 4) {
        // eight warps of one sub-block each on K-split launches that keep their
        // split, at four vectors (token 1566 -> 1579 GB/s; at five their
        // 96-register bound spills)
        if constexpr (NV == 4) {
            const long long tiles = (rows + 63) / 64;
            const int chunks = (int)(cols / PolQ4_K::kChunkCols);
            const Plan p4 = make_plan<PolColSplit<PolQ4_KWide>, NV, 2, false>(dev, tiles, chunks, 0);
            const Plan p8 = make_plan<PolColSplit<PolQ4_KWide8>, NV, 2, false>(dev, tiles, chunks, 0);
            if (p4.ksplit > 1 && p8.ksplit >= p4.ksplit)
                return f(PolColSplit<PolQ4_KWide8>{}, std::integral_constant<int, 2>{});
        }
        // (Q4_K token n_vec 4 / 6 / 8: 1521 / 1192 / 953 -> 1569 / 1247 / 1075
        // GB/s; at n_vec 3 it lost, 1752 -> 1682)
        return f(PolColSplit<PolQ4_KWide>{}, std::integral_constant<int, 2>{});
    } else if constexpr (P::kNibbles && NV <= 2) {
        // column-split stages where the launch does not split K over clusters
        // (enough 64-row tiles to give every CTA slot two): Q4_0 gate|up
        // 28672x4096 3386 -> 3635 GB/s; with a K split they lost (o 4096x4096
        // 1622 -> 1482, down 4096x14336 2877 -> 2413 GB/s).  At two vectors
        // the Q4_0 token gained (2137 -> 2277 GB/s) and the Q4_K token lost
        // (1995 -> 1885), whose decode holds more registers per row; with the
        // run-time pair offset below Q4_K gained too (2000 -> 2030).  With the
        // run-time pair offset below, column split on the K-split launches
        // still lost (Q4_0 token 3157 -> 2715, Q4_K 2572 -> 2397, Q4_0 at
        // two vectors 2398 -> 2289).
        constexpr int TR = 32 * R;
        const bool k_split = (rows + TR - 1) / TR * 2 <= (long long)dev.num_sms * ctas_per_sm<P, NV, R>();
        // The column-split decode takes the warp's pair of blocks at a run-time
        // offset (PolQ4_0Pair, PolQ4_KWide): one copy of it for the four warps
        // instead of four with constant offsets, which the instruction cache
        // held poorly (Q4_0 token 3060 -> 3161 GB/s, gate|up 3652 -> 3813, at
        // two vectors 2320 -> 2399; Q4_K token 2551 -> 2572).  The same change
        // on the Q8_0 one-vector decode lost (8B token 4955 -> 4048 GB/s): its
        // 17 word loads per pair and the rolled loop cost more than the cache,
        // and so did a rolled loop over the pair decodes on the 4-bit formats'
        // K-split launches (Q4_0 token 3149 -> 3092, Q4_K 2572 -> 2497).  A
        // fourth CTA per SM at 72 registers did not change the Q4_0 token.
        if (!k_split) {
            if constexpr (std::is_same<P, PolQ4_0>::value) return f(PolColSplit<PolQ4_0Pair>{}, RT{});
            else return f(PolColSplit<PolQ4_KWide>{}, RT{});
        }
        return f(P{}, RT{});
    } else {
        return f(P{}, RT{});
    }
}

template <class P, int NV>
hq_status dense_nv(const DeviceInfo &dev, const void *W, const void *x, void *y, const int32_t *mult,
                   const int32_t *shift, long long rows, long long cols, const MatvecExtras *lora,
                   cudaStream_t stream) {
    return with_dense_policy<P, NV>(dev, rows, cols, [&](auto pol, auto rt) {
        return dense_nv_r<decltype(pol), NV, decltype(rt)::value>(dev, W, x, y, mult, shift, rows, cols, lora,
                                                                   stream);
    });
}

// Policy identifiers reported by the plan query.
template <class Pol>
constexpr int policy_id() {
    return std::is_same<Pol, PolQ8_0Short>::value ? 1
         : Pol::kColSplit ? 4 : 0;
}

// Test-only: the geometry make_plan gives one dense launch, for a device
// described by `dev` (only num_sms and max_smem_optin are read) and a kernel
// of `regs` registers per thread.
template <class P, int NV>
hq_status dense_plan(const DeviceInfo &dev, long long rows, long long cols, int regs, int64_t *out) {
    return with_dense_policy<P, NV>(dev, rows, cols, [&](auto pol, auto rt) {
        using Pol = decltype(pol);
        constexpr int R = decltype(rt)::value;
        using L = Layout<Pol, NV, R, false>;
        const long long tiles = (rows + L::TR - 1) / L::TR;
        const Plan p = make_plan<Pol, NV, R, false>(dev, tiles, (int)(cols / Pol::kChunkCols), regs);
        out[0] = policy_id<Pol>();
        out[1] = cons_warps<Pol, NV, R>();
        out[2] = L::TR;
        out[3] = p.grid;
        out[4] = p.ksplit;
        out[5] = p.stages;
        out[6] = (int64_t)p.smem;
        out[7] = ctas_per_sm<Pol, NV, R>();
        out[8] = p.slots;
        out[9] = tiles;
        return HQ_OK;
    });
}

template <class P>
hq_status plan_dispatch(const DeviceInfo &dev, long long rows, long long cols, int n_vec, int regs, int64_t *out) {
    switch (n_vec) {
        case 1: return dense_plan<P, 1>(dev, rows, cols, regs, out);
        case 2: return dense_plan<P, 2>(dev, rows, cols, regs, out);
        case 3: return dense_plan<P, 3>(dev, rows, cols, regs, out);
        case 4: return dense_plan<P, 4>(dev, rows, cols, regs, out);
        case 5: return dense_plan<P, 5>(dev, rows, cols, regs, out);
        case 6: return dense_plan<P, 6>(dev, rows, cols, regs, out);
        case 7: return dense_plan<P, 7>(dev, rows, cols, regs, out);
        case 8: return dense_plan<P, 8>(dev, rows, cols, regs, out);
        default: return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    }
}

template <class P>
hq_status dense_dispatch(const DeviceInfo &dev, const void *W, const void *x, void *y,
                         const int32_t *mult, const int32_t *shift, long long rows, long long cols,
                         int n_vec, const MatvecExtras *lora, cudaStream_t stream) {
    switch (n_vec) {
        case 1: return dense_nv<P, 1>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 2: return dense_nv<P, 2>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 3: return dense_nv<P, 3>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 4: return dense_nv<P, 4>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 5: return dense_nv<P, 5>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 6: return dense_nv<P, 6>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 7: return dense_nv<P, 7>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        case 8: return dense_nv<P, 8>(dev, W, x, y, mult, shift, rows, cols, lora, stream);
        default: return set_error(HQ_ERR_NVEC, "n_vec %d not in [1,8]", n_vec);
    }
}

template <int NVMAX>
hq_status moe_nv(const DeviceInfo &dev, const void *W_bank, const int32_t *ids, const float *x,
                 int x_per_slot, float *y, long long n_experts, int n_active, long long rows,
                 long long cols, int n_vec, const MoeEpi &epi, cudaStream_t stream) {
    using P = typename std::conditional<NVMAX == 1, PolQ8_0Moe, PolQ8_0>::type;
    constexpr int R = 1;
    KArgs a = {};
    const long long row_bytes = cols / 32 * P::kBlockBytes;
    hq_status st = encode_2d(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, W_bank, (uint64_t)(row_bytes / 4),
                             (uint64_t)(rows * n_experts), (uint64_t)row_bytes, P::kBoxInner, 32 * R, false);
    if (st != HQ_OK) return st;
    a.y = y;
    a.x = x;
    a.ids = ids;
    a.fault = dev.fault;
    a.rows = rows;
    a.cols = cols;
    a.n_experts = n_experts;
    a.n_chunks = (int)(cols / P::kChunkCols);
    a.num_tiles = (int)((rows + 32 * R - 1) / (32 * R));
    a.n_vec = n_vec;
    a.n_active = n_active;
    a.x_per_slot = x_per_slot;
    a.moe_epi = epi.kind;
    a.router_w = epi.router_w;
    a.ids_ready = epi.ids_ready;
    if (epi.kind == kEpiCombine) {
        // G CTAs per row tile over the tile's expert groups: the largest G
        // (at most kCombineCluster) whose clusters all fit in one wave, as the
        // occupancy calculator counts them (clusters are placed within a GPC)
        const int regs = kernel_regs<P, NVMAX, R, true>();
        Plan p = make_plan<P, NVMAX, R, true>(dev, a.num_tiles, a.n_chunks, regs, 1);
        for (int G = kCombineCluster; G > 1; --G) {
            const Plan q = make_plan<P, NVMAX, R, true>(dev, (long long)a.num_tiles * G, a.n_chunks, regs, G);
            if (max_active_clusters<P, NVMAX, R, true>(dev, G, q.smem) >= a.num_tiles) {
                p = q;
                break;
            }
        }
        return launch_tma<P, NVMAX, R, true>(a, p, stream);
    }
    // The group count is only known on the device; plan for the most groups the
    // pairs can form (every pair its own expert, at most n_experts of them).
    const long long max_groups = std::min<long long>((long long)n_vec * n_active,
                                                     n_experts * (((long long)n_vec * n_active + NVMAX - 1) / NVMAX));
    Plan p = make_plan<P, NVMAX, R, true>(dev, (long long)a.num_tiles * max_groups, a.n_chunks,
                                          kernel_regs<P, NVMAX, R, true>());
    if (p.ksplit > 1) p.grid = (int)((long long)a.num_tiles * max_groups * p.ksplit);
    return launch_tma<P, NVMAX, R, true>(a, p, stream);
}

}  // namespace

// The public launchers are compiled in five parts (HQ_PART 0..4, one object
// file each) so that the template instantiations build in parallel.
#if !defined(HQ_PART) || HQ_PART == 0 || HQ_PART == 1 || HQ_PART == 4
// the float format of this part: Q8_0 (part 0), Q4_0 (part 1), Q4_K (part 4)
using PartPol = std::conditional<HQ_PART == 1, PolQ4_0, std::conditional<HQ_PART == 4, PolQ4_K, PolQ8_0>::type>::type;

hq_status HQ_PART_NAME(launch_matvec_float)(const void *W, const float *x, float *y, int64_t rows,
                                            int64_t cols, int n_vec, const MatvecExtras *lora,
                                            cudaStream_t stream) {
    constexpr int FMT = (HQ_PART == 1) ? 1 : 0;
    using P = PartPol;
    DeviceInfo *dev = nullptr;
    hq_status st = device_info(&dev);
    if (st != HQ_OK) return st;
    if (cols % 256 == 0) return dense_dispatch<P>(*dev, W, x, y, nullptr, nullptr, rows, cols, n_vec, lora, stream);
    if (HQ_PART == 4) return set_error(HQ_ERR_SHAPE, "Q4_K needs cols %% 256 == 0 (cols = %lld)", (long long)cols);
    const unsigned grid = (unsigned)((rows + 7) / 8);
    const MatvecExtras none;
    const MatvecExtras &l = lora ? *lora : none;
    note_launch();
    matvec_plain_kernel<FMT><<<grid, 256, 0, stream>>>((const uint8_t *)W, x, y, rows, cols, n_vec,
                                                       l.B, l.u, l.scale, l.rank);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "matvec launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}
#endif

#if !defined(HQ_PART) || HQ_PART == 0 || HQ_PART == 1 || HQ_PART == 4
hq_status HQ_PART_NAME(debug_plan_float)(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin,
                                         int regs, int64_t *out) {
    using P = PartPol;
    DeviceInfo dev;
    dev.num_sms = num_sms;
    dev.max_smem_optin = smem_optin;
    return plan_dispatch<P>(dev, rows, cols, n_vec, regs, out);
}
#endif

#if HQ_PART == 2
hq_status debug_plan_i8(int n_vec, int64_t rows, int64_t cols, int num_sms, int smem_optin, int regs,
                        int64_t *out) {
    DeviceInfo dev;
    dev.num_sms = num_sms;
    dev.max_smem_optin = smem_optin;
    return plan_dispatch<PolI8>(dev, rows, cols, n_vec, regs, out);
}

hq_status launch_matvec_i8(const int8_t *W, const int8_t *x, const int32_t *mult,
                           const int32_t *shift, int8_t *y, int64_t rows, int64_t cols, int n_vec,
                           cudaStream_t stream) {
    DeviceInfo *dev = nullptr;
    hq_status st = device_info(&dev);
    if (st != HQ_OK) return st;
    if (cols % 128 == 0)
        return dense_dispatch<PolI8>(*dev, W, x, y, mult, shift, rows, cols, n_vec, nullptr, stream);
    note_launch();
    matvec_i8_plain_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(W, x, mult, shift, y, rows, cols, n_vec);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "int8 matvec launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}

hq_status launch_lora_down(const uint16_t *A, const float *x, float *u, int rank, int64_t cols,
                           int n_vec, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rank, 1, 1);
    cfg.blockDim = dim3(kLoraThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lora_down_kernel, A, x, u, rank, (long long)cols, n_vec);
    if (e == cudaSuccess) note_launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "adapter launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}

hq_status launch_wait_timeout_selftest(uint32_t *fault, int64_t cycles, cudaStream_t stream) {
    note_launch();
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(fault, (long long)cycles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "self-test launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}

hq_status launch_requant_debug(const int32_t *acc, const int32_t *mult, const int32_t *shift,
                               int8_t *y, int64_t n, int64_t rows, cudaStream_t stream) {
    const long long blocks = std::min<long long>((n + 255) / 256, 65535);
    note_launch();
    requant_debug_kernel<<<(unsigned)std::max<long long>(blocks, 1), 256, 0, stream>>>(acc, mult, shift, y, n, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(HQ_ERR_LAUNCH, "requant launch: %s", cudaGetErrorString(e));
    return HQ_OK;
}
#endif

#if HQ_PART == 3
hq_status launch_moe_q8_0(const void *W_bank, const int32_t *ids, const float *x, int x_per_slot,
                          float *y, int64_t n_experts, int n_active, int64_t rows, int64_t cols,
                          int n_vec, const MoeEpi *epi, cudaStream_t stream) {
    const MoeEpi none;
    const MoeEpi &e = epi ? *epi : none;
    DeviceInfo *dev = nullptr;
    hq_status st = device_info(&dev);
    if (st != HQ_OK) return st;
    if ((long long)n_vec * n_active > kMaxPairs)
        return set_error(HQ_ERR_SHAPE, "n_vec * n_active = %lld exceeds %d",
                         (long long)n_vec * n_active, kMaxPairs);
    if (cols % 256 != 0)
        return set_error(HQ_ERR_SHAPE, "MoE needs cols %% 256 == 0 (cols = %lld)", (long long)cols);
    if (n_vec <= 1) return moe_nv<1>(*dev, W_bank, ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec, e, stream);
    if (n_vec <= 2) return moe_nv<2>(*dev, W_bank, ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec, e, stream);
    if (n_vec <= 4) return moe_nv<4>(*dev, W_bank, ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec, e, stream);
    return moe_nv<8>(*dev, W_bank, ids, x, x_per_slot, y, n_experts, n_active, rows, cols, n_vec, e, stream);
}
#endif

}  // namespace hq
