// quant.cu -- online fine-grained E4M3 quantizers (HBM-bound).
//
// One FP32 scale per group, computed from the current group only:
// s = fl32(amax / 448), codes = E4M3_RNE_satfinite(fl32(x / s)), both
// divisions IEEE round-to-nearest.  A zero scale stores 0 and codes that keep
// only the sign of x.
//   * 1x128 tiles per token per 128 channels, and 128x128 weight blocks:
//     DeepSeek-V3 FP8 post (innerforce.co.kr), fine-grained quantization,
//     Figure 7 (a).
//   * Scales from the current tensor, no history: "Unified E4M3 format in
//     DeepSeek-V3" (codingmall.com), Dynamic Scaling and Online Quantization.
//   * 128x1 token-axis groups with a transposed (K-major) output for the
//     weight-gradient GEMM, whose reduction runs over tokens: "DeepSeek FP8
//     Training" (arcalunar.github.io), backward pass, Wgrad step 1.
//   * Both of the above from one read of the BF16 tensor (the activation is
//     cached in FP8 for the backward pass: DeepSeek-V3 FP8 post, low-precision
//     storage paragraph): quant_act_dual_kernel.
#include <cuda_runtime.h>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8fg {
namespace {

// bf16_lo / bf16_hi, GroupScale (the division by the group scale),
// quant4 / quant_quad / quant_quad_bf16 (four values to four codes) and
// quad_amax_bf16: quant_math.cuh, shared with the GEMM's fused activation
// quantizer so that both write the same codes.

// ------------------------------------------------------------ 1 x 128 ----
// Grid (row blocks, 128-column groups): a CTA owns kRowsPerCta rows of one
// group column c.  A lane quad owns one row's group (4 lanes x 32 BF16 = 256
// bytes): lane j of the quad loads the group's 16-byte chunks 2j, 2j+1,
// 2j+8, 2j+9, so that its 32 codes are two 16-byte runs of the output row
// (one 16-byte store each); the group maximum needs two shuffles, and the
// scale's division and reciprocal are shared by 32 elements per lane.  A warp
// covers 8 rows per step and keeps kRowU steps' loads in flight; the scales
// of consecutive rows are contiguous in scales[c * rows + r].
constexpr int kRowU = 2;
constexpr int kRowsPerCta = 64 * kRowU;

__global__ void __launch_bounds__(256) quant_act_rows_kernel(const uint4* __restrict__ x, int64_t rows,
                                                             int64_t cols, uint4* __restrict__ q,
                                                             float* __restrict__ scales) {
    const int64_t c = blockIdx.y;
    const int j = threadIdx.x & 3;        // chunks 2j, 2j+1, 2j+8, 2j+9 of the group
    const int rq = threadIdx.x >> 2;      // row of the quad within a 64-row step
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + rq;
    uint4 v[kRowU][4];
#pragma unroll
    for (int u = 0; u < kRowU; ++u) {
        const int64_t r = r0 + 64 * u;
        const uint4* src = x + (r * cols + c * kGroup) / 8 + 2 * j;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[u][k] = make_uint4(0, 0, 0, 0);
            if (r < rows) v[u][k] = __ldcs(src + (k & 1) + 8 * (k >> 1));
        }
    }
#pragma unroll
    for (int u = 0; u < kRowU; ++u) {
        const int64_t r = r0 + 64 * u;
        const float amax = quad_amax_bf16(v[u]);
        if (r >= rows) continue;
        const float s = __fdiv_rn(amax, 448.0f);
        const GroupScale gs(s);
        uint4* dst = q + (r * cols + c * kGroup) / 16 + j;
        with_mode(gs, [&](auto md) {
            constexpr int kM = decltype(md)::value;
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // chunks 2j + 8h and 2j + 8h + 1
                uint4 out;
                out.x = quant_quad_bf16<kM>(v[u][2 * h].x, v[u][2 * h].y, gs);
                out.y = quant_quad_bf16<kM>(v[u][2 * h].z, v[u][2 * h].w, gs);
                out.z = quant_quad_bf16<kM>(v[u][2 * h + 1].x, v[u][2 * h + 1].y, gs);
                out.w = quant_quad_bf16<kM>(v[u][2 * h + 1].z, v[u][2 * h + 1].w, gs);
                __stcs(dst + 4 * h, out);
            }
        });
        if (j == 0) scales[c * rows + r] = s;
    }
}

// ------------------------------------------------------------ 128 x 1 ----
// A CTA owns a tile of 128 tokens x 64 channels.  The BF16 tile is staged in
// shared memory (rows of 32 words + 1 pad word: conflict-free both ways),
// each thread reduces 16 tokens of a channel pair, the 8 partial maxima meet
// in shared memory, and each thread writes 16 codes per channel as one
// 16-byte store into the transposed output q[cols, rows].
constexpr int kColTileC = 64;

__global__ void __launch_bounds__(256) quant_act_cols_kernel(const uint4* __restrict__ x, int64_t rows,
                                                             int64_t cols, uint8_t* __restrict__ q,
                                                             float* __restrict__ scales) {
    __shared__ uint32_t tile[kGroup][kColTileC / 2 + 1];
    __shared__ float part[8][kColTileC];
    const int t = threadIdx.x;
    const int64_t n_tb = rows / kGroup;
    const int64_t n_cb = (cols + kColTileC - 1) / kColTileC;
    for (int64_t tid = blockIdx.x; tid < n_tb * n_cb; tid += gridDim.x) {
        const int64_t tb = tid % n_tb, cb = tid / n_tb;
        const int64_t r0 = tb * kGroup, c0 = cb * kColTileC;
        // load: 8 lanes x 16 bytes per row, 32 rows per pass, 4 passes
        uint4 v[4];
        const int vcol = (t & 7) * 8;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = (t >> 3) + 32 * p;
            v[p] = make_uint4(0, 0, 0, 0);
            if (c0 + vcol < cols) v[p] = __ldcs(x + ((r0 + r) * cols + c0 + vcol) / 8);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = (t >> 3) + 32 * p;
            uint32_t* dst = &tile[r][(t & 7) * 4];
            dst[0] = v[p].x;
            dst[1] = v[p].y;
            dst[2] = v[p].z;
            dst[3] = v[p].w;
        }
        __syncthreads();
        const int cp = t & 31;  // channel pair: channels 2cp, 2cp+1 of the tile
        const int rs = t >> 5;  // token segment: tokens 16rs .. 16rs+15
        float lo[16], hi[16];
        float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const uint32_t w = tile[16 * rs + r][cp];
            lo[r] = bf16_lo(w);
            hi[r] = bf16_hi(w);
            a0 = fmaxf(a0, fabsf(lo[r]));
            a1 = fmaxf(a1, fabsf(hi[r]));
        }
        part[rs][2 * cp] = a0;
        part[rs][2 * cp + 1] = a1;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            a0 = fmaxf(a0, part[k][2 * cp]);
            a1 = fmaxf(a1, part[k][2 * cp + 1]);
        }
        const float s0 = __fdiv_rn(a0, 448.0f), s1 = __fdiv_rn(a1, 448.0f);
        const GroupScale g0(s0), g1(s1);
        const int64_t ch0 = c0 + 2 * cp;
        if (ch0 < cols) {
            with_mode(g0, [&](auto md) {
                constexpr int kM = decltype(md)::value;
                uint4 o;
                o.x = quant_quad<kM>(lo[0], lo[1], lo[2], lo[3], g0);
                o.y = quant_quad<kM>(lo[4], lo[5], lo[6], lo[7], g0);
                o.z = quant_quad<kM>(lo[8], lo[9], lo[10], lo[11], g0);
                o.w = quant_quad<kM>(lo[12], lo[13], lo[14], lo[15], g0);
                __stcs(reinterpret_cast<uint4*>(q + ch0 * rows + r0 + 16 * rs), o);
            });
            if (rs == 0) scales[tb * cols + ch0] = s0;
        }
        if (ch0 + 1 < cols) {
            with_mode(g1, [&](auto md) {
                constexpr int kM = decltype(md)::value;
                uint4 o;
                o.x = quant_quad<kM>(hi[0], hi[1], hi[2], hi[3], g1);
                o.y = quant_quad<kM>(hi[4], hi[5], hi[6], hi[7], g1);
                o.z = quant_quad<kM>(hi[8], hi[9], hi[10], hi[11], g1);
                o.w = quant_quad<kM>(hi[12], hi[13], hi[14], hi[15], g1);
                __stcs(reinterpret_cast<uint4*>(q + (ch0 + 1) * rows + r0 + 16 * rs), o);
            });
            if (rs == 0) scales[tb * cols + ch0 + 1] = s1;
        }
        __syncthreads();  // tile and part are reused by the next tile
    }
}

// ------------------------------------------------- 1 x 128 and 128 x 1 ----
// One CTA per 128 x 128 tile of X, 256 threads.  A lane quad owns one row's
// 1x128 group in each of two passes (rows q and q + 64 for quad q): lane j
// loads the group's 16-byte chunks 2j, 2j+1, 2j+8, 2j+9 into registers, so
// that its 32 codes form two 16-byte runs of the output row (16-byte stores)
// and the group's amax, division and reciprocal are shared by 32 elements
// per lane.  The row pass quantizes from those registers; the same registers
// are written to a shared tile (rows of 64 words + 4 pad words: the two rows
// of a quarter-warp's 16-byte stores fall on disjoint banks, and a warp
// reading 32 consecutive words of one row is conflict-free) for the column
// pass, which gives thread t the channel pair t % 64 over 32 tokens (t / 64);
// the 4 partial maxima meet in shared memory, and each thread writes 2 x 16
// codes per channel into q_col_t[cols, rows].  The arithmetic is the same as
// the single-axis kernels', so both outputs equal theirs bit for bit.
constexpr int kTileWords = kGroup / 2 + 4;   // padded row of the shared tile

__global__ void __launch_bounds__(256, 4) quant_act_dual_kernel(const uint4* __restrict__ x, int64_t rows,
                                                                int64_t cols, uint4* __restrict__ q_row,
                                                                float* __restrict__ s_row,
                                                                uint8_t* __restrict__ q_col_t,
                                                                float* __restrict__ s_col) {
    __shared__ __align__(16) uint32_t tile[kGroup][kTileWords];
    __shared__ float part[4][kGroup];
    const int t = threadIdx.x;
    const int j = t & 3;        // lane of the quad
    const int rq = t >> 2;      // quad: rows rq and rq + 64 of the tile
    const int64_t tb = blockIdx.x, cb = blockIdx.y;
    const int64_t r0 = tb * kGroup, c0 = cb * kGroup;
    uint4 v[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint4* src = x + ((r0 + rq + 64 * u) * cols + c0) / 8 + 2 * j;
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = __ldcs(src + (k & 1) + 8 * (k >> 1));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint4*>(&tile[rq + 64 * u][4 * (2 * j + (k & 1) + 8 * (k >> 1))]) = v[u][k];
    {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t r = r0 + rq + 64 * u;
            const float amax = quad_amax_bf16(v[u]);
            const float s = __fdiv_rn(amax, 448.0f);
            const GroupScale gs(s);
            uint4 lo, hi;   // codes of chunks 2j, 2j+1 and of chunks 2j+8, 2j+9
            with_mode(gs, [&](auto md) {
                constexpr int kM = decltype(md)::value;
                lo.x = quant_quad_bf16<kM>(v[u][0].x, v[u][0].y, gs);
                lo.y = quant_quad_bf16<kM>(v[u][0].z, v[u][0].w, gs);
                lo.z = quant_quad_bf16<kM>(v[u][1].x, v[u][1].y, gs);
                lo.w = quant_quad_bf16<kM>(v[u][1].z, v[u][1].w, gs);
                hi.x = quant_quad_bf16<kM>(v[u][2].x, v[u][2].y, gs);
                hi.y = quant_quad_bf16<kM>(v[u][2].z, v[u][2].w, gs);
                hi.z = quant_quad_bf16<kM>(v[u][3].x, v[u][3].y, gs);
                hi.w = quant_quad_bf16<kM>(v[u][3].z, v[u][3].w, gs);
            });
            uint4* dst = q_row + (r * cols + c0) / 16 + j;
            __stcs(dst, lo);
            __stcs(dst + 4, hi);
            if (j == 0) s_row[cb * rows + r] = s;
        }
    }
    __syncthreads();
    const int cp = t & 63;   // channel pair: channels 2cp, 2cp+1 of the tile
    const int rs = t >> 6;   // token segment: tokens 32rs .. 32rs+31
    uint32_t w[32];          // the segment's words, read once for the maximum and the codes
#pragma unroll
    for (int r = 0; r < 32; ++r) w[r] = tile[32 * rs + r][cp];
    uint32_t m2 = 0;         // both channels' maxima as 16-bit patterns
#pragma unroll
    for (int r = 0; r < 32; ++r) m2 = __vmaxu2(m2, w[r] & 0x7FFF7FFFu);
    part[rs][2 * cp] = __uint_as_float(m2 << 16);
    part[rs][2 * cp + 1] = __uint_as_float(m2 & 0xFFFF0000u);
    __syncthreads();
    float a0 = part[0][2 * cp], a1 = part[0][2 * cp + 1];
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        a0 = fmaxf(a0, part[k][2 * cp]);
        a1 = fmaxf(a1, part[k][2 * cp + 1]);
    }
    const float s0 = __fdiv_rn(a0, 448.0f), s1 = __fdiv_rn(a1, 448.0f);
    const GroupScale g0(s0), g1(s1);
    const int64_t ch0 = c0 + 2 * cp;
    uint4* dst0 = reinterpret_cast<uint4*>(q_col_t + ch0 * rows + r0 + 32 * rs);
    uint4* dst1 = reinterpret_cast<uint4*>(q_col_t + (ch0 + 1) * rows + r0 + 32 * rs);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t* wk = w + 16 * k;
        // channel 2cp: the low halves of four consecutive tokens' words
        with_mode(g0, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_lo(wk[0]), bf16_lo(wk[1]), bf16_lo(wk[2]), bf16_lo(wk[3]), g0);
            o.y = quant_quad<kM>(bf16_lo(wk[4]), bf16_lo(wk[5]), bf16_lo(wk[6]), bf16_lo(wk[7]), g0);
            o.z = quant_quad<kM>(bf16_lo(wk[8]), bf16_lo(wk[9]), bf16_lo(wk[10]), bf16_lo(wk[11]), g0);
            o.w = quant_quad<kM>(bf16_lo(wk[12]), bf16_lo(wk[13]), bf16_lo(wk[14]), bf16_lo(wk[15]), g0);
            __stcs(dst0 + k, o);
        });
        with_mode(g1, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_hi(wk[0]), bf16_hi(wk[1]), bf16_hi(wk[2]), bf16_hi(wk[3]), g1);
            o.y = quant_quad<kM>(bf16_hi(wk[4]), bf16_hi(wk[5]), bf16_hi(wk[6]), bf16_hi(wk[7]), g1);
            o.z = quant_quad<kM>(bf16_hi(wk[8]), bf16_hi(wk[9]), bf16_hi(wk[10]), bf16_hi(wk[11]), g1);
            o.w = quant_quad<kM>(bf16_hi(wk[12]), bf16_hi(wk[13]), bf16_hi(wk[14]), bf16_hi(wk[15]), g1);
            __stcs(dst1 + k, o);
        });
    }
    if (rs == 0) {
        s_col[tb * cols + ch0] = s0;
        s_col[tb * cols + ch0 + 1] = s1;
    }
}

// ------------------------------------- 1 x 128 and 128 x 1, staged tile ----
// The same outputs as quant_act_dual_kernel, for large tensors (at least
// kDualStagedTilesPerSm tiles per SM: X[8192,7168] 49.1 against 51.1 us
// back to back, while on X[4096,7168] the register kernel's four CTAs per SM
// give fuller rounds of tiles, 26.4 against 27.2 us).  One CTA per
// 128 x 128 tile of X, 256 threads, 5 CTAs per SM.  The tile is
// copied into shared memory with cp.async (rows of 64 words + 4 pad words;
// no registers held while the copies are in flight, so an SM keeps 160 KB
// of loads in flight), and both passes read it there.  Row pass: a lane quad
// owns one row's 1x128 group in each of two rounds (rows q and q + 64 for
// quad q); lane j takes the group's 16-byte chunks 2j, 2j+1, 2j+8, 2j+9, so
// that its 32 codes form two 16-byte runs of the output row (16-byte
// stores) and the group's amax, division and reciprocal are shared by 32
// elements per lane (the pad puts the two rows of a quarter-warp's 16-byte
// loads on disjoint banks).  Column pass: thread t takes the channel pair
// t % 64 over 32 tokens (t / 64), a warp reading 32 consecutive words of one
// row; the 4 partial maxima meet in shared memory, and each thread writes
// 2 x 16 codes per channel into q_col_t[cols, rows].  The arithmetic is the
// same as the single-axis kernels', so both outputs equal theirs bit for bit.
constexpr int kDualStagedTilesPerSm = 16;

__global__ void __launch_bounds__(256, 5) quant_act_dual_staged_kernel(const uint4* __restrict__ x, int64_t rows,
                                                                       int64_t cols, uint4* __restrict__ q_row,
                                                                       float* __restrict__ s_row,
                                                                       uint8_t* __restrict__ q_col_t,
                                                                       float* __restrict__ s_col) {
    __shared__ __align__(16) uint32_t tile[kGroup][kTileWords];
    __shared__ float part[4][kGroup];
    const int t = threadIdx.x;
    const int64_t tb = blockIdx.x, cb = blockIdx.y;
    const int64_t r0 = tb * kGroup, c0 = cb * kGroup;
    {
        const int l16 = t & 15, hw = t >> 4;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int r = hw + 16 * u;
            cp_async_16(smem_u32(&tile[r][4 * l16]), x + ((r0 + r) * cols + c0) / 8 + l16);
        }
        cp_async_wait_all();
        __syncthreads();
    }
    {
        const int j = t & 3;     // lane of the quad
        const int rq = t >> 2;   // quad: rows rq and rq + 64 of the tile
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t r = r0 + rq + 64 * u;
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[k] = *reinterpret_cast<const uint4*>(&tile[rq + 64 * u][4 * (2 * j + (k & 1) + 8 * (k >> 1))]);
            const float amax = quad_amax_bf16(v);
            const float s = __fdiv_rn(amax, 448.0f);
            const GroupScale gs(s);
            uint4 lo, hi;   // codes of chunks 2j, 2j+1 and of chunks 2j+8, 2j+9
            with_mode(gs, [&](auto md) {
                constexpr int kM = decltype(md)::value;
                lo.x = quant_quad_bf16<kM>(v[0].x, v[0].y, gs);
                lo.y = quant_quad_bf16<kM>(v[0].z, v[0].w, gs);
                lo.z = quant_quad_bf16<kM>(v[1].x, v[1].y, gs);
                lo.w = quant_quad_bf16<kM>(v[1].z, v[1].w, gs);
                hi.x = quant_quad_bf16<kM>(v[2].x, v[2].y, gs);
                hi.y = quant_quad_bf16<kM>(v[2].z, v[2].w, gs);
                hi.z = quant_quad_bf16<kM>(v[3].x, v[3].y, gs);
                hi.w = quant_quad_bf16<kM>(v[3].z, v[3].w, gs);
            });
            uint4* dst = q_row + (r * cols + c0) / 16 + j;
            __stcs(dst, lo);
            __stcs(dst + 4, hi);
            if (j == 0) s_row[cb * rows + r] = s;
        }
    }
    const int cp = t & 63;   // channel pair: channels 2cp, 2cp+1 of the tile
    const int rs = t >> 6;   // token segment: tokens 32rs .. 32rs+31
    uint32_t m2 = 0;         // both channels' maxima as 16-bit patterns
#pragma unroll
    for (int r = 0; r < 32; ++r) m2 = __vmaxu2(m2, tile[32 * rs + r][cp] & 0x7FFF7FFFu);
    part[rs][2 * cp] = __uint_as_float(m2 << 16);
    part[rs][2 * cp + 1] = __uint_as_float(m2 & 0xFFFF0000u);
    __syncthreads();
    float a0 = part[0][2 * cp], a1 = part[0][2 * cp + 1];
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        a0 = fmaxf(a0, part[k][2 * cp]);
        a1 = fmaxf(a1, part[k][2 * cp + 1]);
    }
    const float s0 = __fdiv_rn(a0, 448.0f), s1 = __fdiv_rn(a1, 448.0f);
    const GroupScale g0(s0), g1(s1);
    const int64_t ch0 = c0 + 2 * cp;
    uint4* dst0 = reinterpret_cast<uint4*>(q_col_t + ch0 * rows + r0 + 32 * rs);
    uint4* dst1 = reinterpret_cast<uint4*>(q_col_t + (ch0 + 1) * rows + r0 + 32 * rs);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t wk[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) wk[r] = tile[32 * rs + 16 * k + r][cp];
        // channel 2cp: the low halves of four consecutive tokens' words
        with_mode(g0, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_lo(wk[0]), bf16_lo(wk[1]), bf16_lo(wk[2]), bf16_lo(wk[3]), g0);
            o.y = quant_quad<kM>(bf16_lo(wk[4]), bf16_lo(wk[5]), bf16_lo(wk[6]), bf16_lo(wk[7]), g0);
            o.z = quant_quad<kM>(bf16_lo(wk[8]), bf16_lo(wk[9]), bf16_lo(wk[10]), bf16_lo(wk[11]), g0);
            o.w = quant_quad<kM>(bf16_lo(wk[12]), bf16_lo(wk[13]), bf16_lo(wk[14]), bf16_lo(wk[15]), g0);
            __stcs(dst0 + k, o);
        });
        with_mode(g1, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_hi(wk[0]), bf16_hi(wk[1]), bf16_hi(wk[2]), bf16_hi(wk[3]), g1);
            o.y = quant_quad<kM>(bf16_hi(wk[4]), bf16_hi(wk[5]), bf16_hi(wk[6]), bf16_hi(wk[7]), g1);
            o.z = quant_quad<kM>(bf16_hi(wk[8]), bf16_hi(wk[9]), bf16_hi(wk[10]), bf16_hi(wk[11]), g1);
            o.w = quant_quad<kM>(bf16_hi(wk[12]), bf16_hi(wk[13]), bf16_hi(wk[14]), bf16_hi(wk[15]), g1);
            __stcs(dst1 + k, o);
        });
    }
    if (rs == 0) {
        s_col[tb * cols + ch0] = s0;
        s_col[tb * cols + ch0 + 1] = s1;
    }
}

// ------------------------------------------------------------ 128 x 1 ----
// The 128x1 quantizer alone when cols is a multiple of 128: one CTA per
// 128 x 128 tile, 256 threads, 5 CTAs per SM.  The tile (32 KB) is copied
// into shared memory with cp.async (no registers held while the copies are
// in flight; with no row pass to feed, this beats staging the tile through
// registers), then the column pass of quant_act_dual_kernel: thread t takes
// the channel pair t % 64 over 32 tokens (t / 64), the 4 partial maxima meet
// in shared memory, and each thread writes 2 x 16 codes per channel into
// q_col_t[cols, rows].  A warp always reads 32 consecutive words of one row,
// so the unpadded tile has no bank conflicts.
__global__ void __launch_bounds__(256, 5) quant_act_cols_tile_kernel(const uint4* __restrict__ x, int64_t rows,
                                                                   int64_t cols, uint8_t* __restrict__ q_col_t,
                                                                   float* __restrict__ s_col) {
    __shared__ __align__(16) uint32_t tile[kGroup][kGroup / 2];
    __shared__ float part[4][kGroup];
    const int t = threadIdx.x, l16 = t & 15, hw = t >> 4;
    const int64_t tb = blockIdx.x, cb = blockIdx.y;
    const int64_t r0 = tb * kGroup, c0 = cb * kGroup;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int r = hw + 16 * u;
        cp_async_16(smem_u32(&tile[r][4 * l16]), x + ((r0 + r) * cols + c0) / 8 + l16);
    }
    cp_async_wait_all();
    __syncthreads();
    const int cp = t & 63;   // channel pair: channels 2cp, 2cp+1 of the tile
    const int rs = t >> 6;   // token segment: tokens 32rs .. 32rs+31
    uint32_t m2 = 0;         // both channels' maxima as 16-bit patterns
#pragma unroll
    for (int r = 0; r < 32; ++r) m2 = __vmaxu2(m2, tile[32 * rs + r][cp] & 0x7FFF7FFFu);
    part[rs][2 * cp] = __uint_as_float(m2 << 16);
    part[rs][2 * cp + 1] = __uint_as_float(m2 & 0xFFFF0000u);
    __syncthreads();
    float a0 = part[0][2 * cp], a1 = part[0][2 * cp + 1];
#pragma unroll
    for (int k = 1; k < 4; ++k) {
        a0 = fmaxf(a0, part[k][2 * cp]);
        a1 = fmaxf(a1, part[k][2 * cp + 1]);
    }
    const float s0 = __fdiv_rn(a0, 448.0f), s1 = __fdiv_rn(a1, 448.0f);
    const GroupScale g0(s0), g1(s1);
    const int64_t ch0 = c0 + 2 * cp;
    uint4* dst0 = reinterpret_cast<uint4*>(q_col_t + ch0 * rows + r0 + 32 * rs);
    uint4* dst1 = reinterpret_cast<uint4*>(q_col_t + (ch0 + 1) * rows + r0 + 32 * rs);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t w[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) w[r] = tile[32 * rs + 16 * k + r][cp];
        // channel 2cp: the low halves of four consecutive tokens' words
        with_mode(g0, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_lo(w[0]), bf16_lo(w[1]), bf16_lo(w[2]), bf16_lo(w[3]), g0);
            o.y = quant_quad<kM>(bf16_lo(w[4]), bf16_lo(w[5]), bf16_lo(w[6]), bf16_lo(w[7]), g0);
            o.z = quant_quad<kM>(bf16_lo(w[8]), bf16_lo(w[9]), bf16_lo(w[10]), bf16_lo(w[11]), g0);
            o.w = quant_quad<kM>(bf16_lo(w[12]), bf16_lo(w[13]), bf16_lo(w[14]), bf16_lo(w[15]), g0);
            __stcs(dst0 + k, o);
        });
        with_mode(g1, [&](auto md) {
            constexpr int kM = decltype(md)::value;
            uint4 o;
            o.x = quant_quad<kM>(bf16_hi(w[0]), bf16_hi(w[1]), bf16_hi(w[2]), bf16_hi(w[3]), g1);
            o.y = quant_quad<kM>(bf16_hi(w[4]), bf16_hi(w[5]), bf16_hi(w[6]), bf16_hi(w[7]), g1);
            o.z = quant_quad<kM>(bf16_hi(w[8]), bf16_hi(w[9]), bf16_hi(w[10]), bf16_hi(w[11]), g1);
            o.w = quant_quad<kM>(bf16_hi(w[12]), bf16_hi(w[13]), bf16_hi(w[14]), bf16_hi(w[15]), g1);
            __stcs(dst1 + k, o);
        });
    }
    if (rs == 0) {
        s_col[tb * cols + ch0] = s0;
        s_col[tb * cols + ch0 + 1] = s1;
    }
}

// ---------------------------------------------------------- 128 x 128 ----
// A CTA of 512 threads owns one 128x128 FP32 block at a time and keeps it in
// registers: thread t holds columns 4(t%32)..+3 of rows 4(t/32)+{0..3} and
// 64 + 4(t/32)+{0..3}.  Block amax: warp shuffles, then 16 partials in
// shared memory.  The optional transposed copy goes through a shared tile of
// 4x4-byte-transposed words.
// (Two CTAs per SM, i.e. at most 64 registers: at 65 the SM holds one CTA
// and the kernel ran a third slower.)
__global__ void __launch_bounds__(512, 2) quant_w_kernel(const float4* __restrict__ w, int64_t rows, int64_t cols,
                                                      uint32_t* __restrict__ q, uint8_t* __restrict__ q_t,
                                                      float* __restrict__ scales) {
    __shared__ float red[16];
    // transposed tile: word w of row c (the block's column c, rows 4w..4w+3)
    // at tq[c][w ^ (c / 4)]: the stores below (lane l writes rows 4l..4l+3 of
    // one word column) and the loads (a warp reads 8 rows whose c / 4 are
    // distinct) then touch 32 distinct banks per instruction
    __shared__ uint32_t tq[kGroup][kGroup / 4];
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int64_t nbr = rows / kGroup, nbc = cols / kGroup;
    // this thread's 32 values of block `b`: rows 4 wid + k and 64 + 4 wid + k, columns 4 lane .. 4 lane + 3
    float4 v[8];
    auto load_block = [&](int64_t b) {
        const int64_t r0 = (b / nbc) * kGroup, c0 = (b % nbc) * kGroup;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t r = r0 + 64 * h + 4 * wid + k;
                v[4 * h + k] = __ldcs(w + (r * cols + c0) / 4 + lane);
            }
    };
    if (blockIdx.x < nbr * nbc) load_block(blockIdx.x);
    for (int64_t blk = blockIdx.x; blk < nbr * nbc; blk += gridDim.x) {
        const int64_t br = blk / nbc, bc = blk - br * nbc;
        const int64_t r0 = br * kGroup, c0 = bc * kGroup;
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            amax = fmaxf(fmaxf(amax, fmaxf(fabsf(v[k].x), fabsf(v[k].y))), fmaxf(fabsf(v[k].z), fabsf(v[k].w)));
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[wid] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int k = 1; k < 16; ++k) amax = fmaxf(amax, red[k]);
        const float s = __fdiv_rn(amax, 448.0f);
        const GroupScale gs(s);
        uint32_t code[8];
        with_mode(gs, [&](auto md) {
            constexpr int kM = decltype(md)::value;
#pragma unroll
            for (int k = 0; k < 8; ++k) code[k] = quant_quad<kM>(v[k].x, v[k].y, v[k].z, v[k].w, gs);
        });
        // the next block's loads go out now (v is free): their latency
        // overlaps this block's stores and barriers
        if (blk + gridDim.x < nbr * nbc) load_block(blk + gridDim.x);
        // 16-byte code stores: the warp's 8 rows of codes (4 bytes per lane
        // and row) go through its own 1 KB of the shared tile (rows 8 wid ..
        // 8 wid + 7 of tq, one 128-byte row each: conflict-free word stores),
        // then each lane reads 16 bytes of one row back and stores them
        {
            uint32_t* stage = &tq[8 * wid][0];
#pragma unroll
            for (int k = 0; k < 8; ++k) stage[32 * k + lane] = code[k];
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k = 4 * u + (lane >> 3);   // staged row: code[k] of every lane
                const uint4 o = *reinterpret_cast<const uint4*>(&stage[32 * k + 4 * (lane & 7)]);
                const int64_t r = r0 + 64 * (k >> 2) + 4 * wid + (k & 3);
                __stcs(reinterpret_cast<uint4*>(q) + (r * cols + c0) / 16 + (lane & 7), o);
            }
        }
        if (t == 0) scales[br * nbc + bc] = s;
        if (q_t != nullptr) {
            __syncthreads();   // every warp has read its staged codes back out of tq
            // transpose each 4x4 byte block: word k holds row k, byte u = column u
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w0 = code[4 * h], w1 = code[4 * h + 1], w2 = code[4 * h + 2], w3 = code[4 * h + 3];
                const uint32_t lo01 = __byte_perm(w0, w1, 0x5140), hi01 = __byte_perm(w0, w1, 0x7362);
                const uint32_t lo23 = __byte_perm(w2, w3, 0x5140), hi23 = __byte_perm(w2, w3, 0x7362);
                // column u word: bytes (row0,u),(row1,u),(row2,u),(row3,u)
                const uint32_t c0w = __byte_perm(lo01, lo23, 0x5410);
                const uint32_t c1w = __byte_perm(lo01, lo23, 0x7632);
                const uint32_t c2w = __byte_perm(hi01, hi23, 0x5410);
                const uint32_t c3w = __byte_perm(hi01, hi23, 0x7632);
                const int rw = (16 * h + wid) ^ lane;  // word along rows (rows 4(16h+wid)..+3), swizzled
                tq[4 * lane + 0][rw] = c0w;
                tq[4 * lane + 1][rw] = c1w;
                tq[4 * lane + 2][rw] = c2w;
                tq[4 * lane + 3][rw] = c3w;
            }
            __syncthreads();
            // q_t row (c0 + j) receives the block's column j: 128 bytes = 32
            // words, a quarter (part) per thread; a warp covers the 8 rows
            // j = 32 (wid % 4) + 4 b + wid / 4 (b < 8), whose j / 4 differ
            const int part = lane & 3;
            const int j = 32 * (wid & 3) + 4 * (lane >> 2) + (wid >> 2);
            const int sw = j >> 2;
            uint4 o0, o1;
            o0.x = tq[j][(8 * part + 0) ^ sw];
            o0.y = tq[j][(8 * part + 1) ^ sw];
            o0.z = tq[j][(8 * part + 2) ^ sw];
            o0.w = tq[j][(8 * part + 3) ^ sw];
            o1.x = tq[j][(8 * part + 4) ^ sw];
            o1.y = tq[j][(8 * part + 5) ^ sw];
            o1.z = tq[j][(8 * part + 6) ^ sw];
            o1.w = tq[j][(8 * part + 7) ^ sw];
            uint4* dst = reinterpret_cast<uint4*>(q_t + (c0 + j) * rows + r0 + 32 * part);
            __stcs(dst, o0);
            __stcs(dst + 1, o1);
        }
        __syncthreads();  // red and tq are reused by the next block
    }
}

}  // namespace

cudaError_t launch_quant_act_rows(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales, int num_sms,
                                  cudaStream_t stream) {
    (void)num_sms;
    const dim3 grid(static_cast<unsigned>((rows + kRowsPerCta - 1) / kRowsPerCta), static_cast<unsigned>(cols / kGroup));
    quant_act_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), rows, cols,
                                                    reinterpret_cast<uint4*>(q), scales);
    return cudaPeekAtLastError();
}

cudaError_t launch_quant_act_cols(const void* x, int64_t rows, int64_t cols, uint8_t* q, float* scales, int num_sms,
                                  cudaStream_t stream) {
    if (cols % kGroup == 0 && cols / kGroup <= 65535) {
        const dim3 grid(static_cast<unsigned>(rows / kGroup), static_cast<unsigned>(cols / kGroup));
        quant_act_cols_tile_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), rows, cols, q, scales);
        return cudaPeekAtLastError();
    }
    const int64_t tiles = (rows / kGroup) * ((cols + kColTileC - 1) / kColTileC);
    int64_t grid = tiles;
    if (grid > static_cast<int64_t>(num_sms) * 8) grid = static_cast<int64_t>(num_sms) * 8;
    quant_act_cols_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(static_cast<const uint4*>(x), rows, cols,
                                                                           q, scales);
    return cudaPeekAtLastError();
}

cudaError_t launch_quant_act_dual(const void* x, int64_t rows, int64_t cols, uint8_t* q_row, float* s_row,
                                  uint8_t* q_col_t, float* s_col, int num_sms, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(rows / kGroup), static_cast<unsigned>(cols / kGroup));
    const int64_t tiles = (rows / kGroup) * (cols / kGroup);
    if (tiles >= static_cast<int64_t>(kDualStagedTilesPerSm) * num_sms)
        quant_act_dual_staged_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), rows, cols,
                                                                reinterpret_cast<uint4*>(q_row), s_row, q_col_t,
                                                                s_col);
    else
        quant_act_dual_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), rows, cols,
                                                         reinterpret_cast<uint4*>(q_row), s_row, q_col_t, s_col);
    return cudaPeekAtLastError();
}

cudaError_t launch_quant_w(const float* w, int64_t rows, int64_t cols, uint8_t* q, uint8_t* q_t, float* scales,
                           int num_sms, cudaStream_t stream) {
    const int64_t blocks = (rows / kGroup) * (cols / kGroup);
    int64_t grid = blocks;
    if (grid > static_cast<int64_t>(num_sms) * 4) grid = static_cast<int64_t>(num_sms) * 4;
    quant_w_kernel<<<static_cast<unsigned>(grid), 512, 0, stream>>>(reinterpret_cast<const float4*>(w), rows, cols,
                                                                    reinterpret_cast<uint32_t*>(q), q_t, scales);
    return cudaPeekAtLastError();
}

}  // namespace fp8fg
