// gemm.cu -- block-scaled FP8 GEMM on sm_103a tensor cores (tcgen05 + TMEM).
//
// D[M, N] = A[M, K] . B[N, K]^T, both operands K-major E4M3 with one FP32
// scale per 128-wide K chunk (per row of A; per 128x128 block or per row of
// B).  For every K chunk c the tensor cores accumulate
//     P = sum_{k in chunk c} a[i, k] b[j, k]        (FP32, in TMEM)
// and the promotion warps fold it into FP32 registers:
//     acc[i, j] += P[i, j] * (sa[c, i] * sb(j, c)).
// Sources: "DeepSeek FP8 Training" (arcalunar.github.io), forward pipeline
// steps 3-4 (tile-based FP8 GEMM, FP32 accumulation, BF16 output) and the
// Wgrad / Dgrad pipelines (FP32 and BF16 outputs); DeepSeek-V3 FP8 post
// (innerforce.co.kr), increased-precision accumulation paragraph (the FP8
// MMA's own accumulation is limited, so partial sums are promoted to FP32
// with the dequantization folded in); "Unified E4M3 format in DeepSeek-V3"
// (codingmall.com), Enhanced Numerical Stability (promotion to FP32 registers
// at fixed intervals; the interval here is one 128-wide group).
//
// Kernel structure (one persistent CTA per SM, 12 warps in 3 warpgroups;
// warpgroup 0 gives registers to the promotion warpgroups with setmaxnreg):
//   warp 0      TMA producer: A tile [128 x 128 B] and B tile [256 x 128 B]
//               per K chunk into a 3-stage shared-memory ring (128-byte
//               swizzle), completing on mbarriers;
//   warp 1      MMA issuer (lane 0 issues, the warp waits): before reusing a
//               TMEM buffer it takes the buffer back from the promotion
//               warps on a named barrier (bar.sync), learns from warp 2 on
//               another named barrier that the chunk's operands have landed,
//               then issues 4 x tcgen05.mma.kind::f8f6f4 (K = 32 each) per
//               chunk into one of two 256-column buffers and commits ONCE, to
//               the chunk's "done" mbarrier, on which both the producer
//               (stage free) and the promotion warps (partial sums ready)
//               wait.  The warp touches no shared memory in this loop: an
//               mbarrier wait in the MMA-issuing warp measured 150-300
//               cycles per chunk even on a completed phase, idling the
//               tensor pipe.  Its loop is kept to the barrier pair, the
//               MMAs and one commit: everything it does between a chunk's
//               last MMA issue and the next chunk's first is time the tensor
//               pipe can idle (a clock64-traced build measured ~700 cycles
//               per chunk for this loop with two commits and per-chunk
//               descriptor arithmetic, against 512 for the MMAs);
//   warp 2      operand watcher: waits for each chunk's "full" mbarrier and
//               meets the MMA warp on a named barrier (bar.red.or carries a
//               failed wait);
//   warp 3      per-row B scales only: copies each chunk's B and A scales
//               from global memory by cp.async into a shared ring of slots
//               of 4 chunks, in an order that lets each promotion thread
//               read its own with 16-byte loads;
//   warps 4-11  promotion: wait for the buffer, tcgen05.ld 8 x 16 columns
//               (the next load in flight while the previous 16 columns are
//               scaled and added with packed FP32 FMAs), hand the buffer back
//               (bar.arrive), and after the tile's last chunk write the
//               128 x 256 outputs through shared memory with TMA stores.  With
//               block B scales the A scales come straight from global memory,
//               four chunks ahead, into registers (a tile's first ones during
//               the previous tile's stores), and the B scales 32 chunks per
//               load, one per lane, broadcast by shuffles; per-row B scales
//               come from warp 3's ring.
// The MMA of chunk c+1 runs while the promotion warps fold chunk c.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8fg {
namespace {

constexpr int BM = 128;   // rows of A per tile (TMEM lanes)
constexpr int BN = 256;   // rows of B per tile (TMEM columns per buffer): 256 or 128
constexpr int NBUF = 512 / BN;   // TMEM accumulator buffers (all 512 columns)
constexpr int ECOLS = BN / 2;    // columns of a tile per promotion thread
constexpr int BK = 128;   // one quantization group along K
constexpr int MMA_K = 32; // K per tcgen05.mma for 8-bit operands
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 128 + 32 * EPI_WARPS;
// registers per thread: 168 at launch (384 x 168 = 64512); after the split
// warpgroup 0 keeps 64 and the two promotion warpgroups take 216 each
// (128 x 64 + 256 x 216 = 63488, within the launch total).
constexpr int REGS_LOW = 64, REGS_HIGH = 216;
constexpr uint32_t TMEM_COLS = NBUF * BN;
constexpr uint32_t A_BYTES = BM * BK;
constexpr uint32_t B_BYTES = BN * BK;
// Named barriers 1 .. NBUF: the 8 promotion warps hand TMEM buffer b back
// to the MMA warp through barrier 1 + b (bar.arrive by them, bar.sync by the
// whole MMA warp).
constexpr int kRelThreads = 32 * (1 + EPI_WARPS);
// Named barrier 1 + NBUF: the operand watcher (warp 2) and the MMA warp meet
// on it once per chunk (bar.red.or: the watcher reports a failed wait).
constexpr int kOpsBar = 1 + NBUF;
constexpr int kOpsThreads = 64;
// MMA completion of chunk g (counted over the CTA's tiles): mbarrier
// done[g % kDone], one commit per chunk.  kDone >= max(stages, NBUF) keeps
// every parity wait on it unambiguous: the next phase of done[g % kDone]
// (chunk g + kDone) cannot complete before the producer and the promotion
// warps have waited for chunk g (the producer has not loaded chunk
// g + kDone's operands yet, and the MMA warp issues it only after the
// promotion warps hand back chunk g + kDone - NBUF >= g).
constexpr uint32_t kDone = 4;
// Limit of the promotion warps' wait for a chunk's commit (see run_epilogue):
// far above the longest settable limit of the other waits.
constexpr uint64_t kHandoffLimitNs = 3 * kMaxWaitLimitNs;
// Limit of the tear-down waits after a failure (copies in flight landing):
// far above a copy's latency; running out records kErrTeardown.
constexpr uint64_t kTeardownLimitNs = 10000000ull;

// Per-row B scales: chunks per slot of the scale ring.  The promotion warps
// wait for a slot and release it once per group of chunks: a build without
// the per-chunk wait, warp vote and arrival (not a correct kernel) ran the
// Wgrad GEMM 17% faster; groups of 4 recover 4% (groups of 2 were slower;
// 8 or 16 chunks per slot, with the 196 KB cap below lifted, no faster).
constexpr int kScaleGroup = 4;

// Shared memory.  kRowB = 1 (B scales per row of B) also keeps a ring of
// the chunks' B scales and A scales, staged by warp 3 (run_scales).  (Three
// operand stages measured faster than four on the Fprop shape: the fourth
// leaves almost no L1 for the scale loads.)
template <int kRowB>
struct __align__(1024) Smem {
    static constexpr int kStages = BN == 256 ? 3 : 4;
    static constexpr int kSlots = kRowB ? 3 : 1;   // per-row scale ring: slots of kScaleGroup chunks
    uint8_t a[kStages][A_BYTES];
    uint8_t b[kStages][B_BYTES];
    uint8_t out[EPI_WARPS][32 * 128];   // per promotion warp: 32 rows x 128 B, 128-byte swizzle
    float sb[kSlots][kRowB ? kScaleGroup : 1][BN];
    float sa[kSlots][kRowB ? kScaleGroup : 1][kRowB ? BM : 4];
    uint64_t full[kStages];
    uint64_t done[kDone];
    uint64_t sfull[kSlots];
    uint64_t sempty[kSlots];
    uint64_t drain;
    uint64_t pfull[5];    // fused A quantization: tile slot loaded (TMA)
    uint64_t pempty[5];   // fused A quantization: tile slot consumed (8 warps)
    uint32_t tmem_base;
    int abort_flag;
};

template <int kRowB>
constexpr size_t smem_bytes() {
    return sizeof(Smem<kRowB>) + 1024;   // + alignment slack of the dynamic buffer
}
// At most 196 KB, so that the carve-out leaves 60 KB of L1 (measured faster
// than the 228 KB carve-out with its 28 KB of L1).
static_assert(smem_bytes<0>() <= 196 * 1024 && smem_bytes<1>() <= 196 * 1024, "shared memory per CTA");
static_assert(kDone == 4 && kDone >= Smem<0>::kStages && kDone >= Smem<1>::kStages && kDone >= NBUF,
              "done ring: a power of two no shorter than the stage ring and the TMEM buffers");

struct Params {
    const float* sa;
    const float* sb;
    int64_t sb_stride_n;
    int64_t sb_stride_k;
    int64_t sb_group_stride;  // grouped: elements between consecutive experts' scale arrays
    int bscale;
    void* d;
    int out_bf16;
    int64_t M, N, K;
    const int32_t* offsets;
    int G;
    int m_fastest;
    int* status;
    uint64_t limit_ns;
    // fused A quantization (fp8_gemm_quant_a): the BF16 A operand, the
    // buffers its codes and scales are written to (the A tensor map and sa
    // read the same ones), and the per-band tile counters
    uint2* qa;
    float* sa_out;
    int* band_flags;
    // ceil(M / 128): a partial last row tile counts.  Passed in rather than
    // computed by the kernel: computing it there changed the register
    // allocation of the promotion warps (80 -> 100 bytes of spill loads,
    // Fprop 2% slower); read from the parameters they spill nothing.
    int64_t m_tiles;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4 (unused for this layout: 1)
//   bits 32-45  stride-dimension byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-48  fixed 0b001
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
FP8FG_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4: D = F32 (bits 4-5 = 1), A = B = E4M3
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

// Tile t -> origin (m0, n0).  Tile counts fit in 32 bits (checked on the
// host), so the divisions stay 32-bit and inline.
FP8FG_DEV void tile_origin(int64_t t, int64_t m_tiles, int64_t n_tiles, int m_fastest, int64_t& m0, int64_t& n0) {
    const uint32_t tt = static_cast<uint32_t>(t);
    if (m_fastest) {
        const uint32_t mt = static_cast<uint32_t>(m_tiles);
        const uint32_t q = tt / mt;
        m0 = static_cast<int64_t>(tt - q * mt) * BM;
        n0 = static_cast<int64_t>(q) * BN;
    } else {
        const uint32_t nt = static_cast<uint32_t>(n_tiles);
        const uint32_t q = tt / nt;
        m0 = static_cast<int64_t>(q) * BM;
        n0 = static_cast<int64_t>(tt - q * nt) * BN;
    }
}

// Expert owning row m0: the g with offsets[g] <= m0 < offsets[g+1].
FP8FG_DEV int expert_of(const int32_t* offsets, int G, int64_t m0) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(__ldg(offsets + mid)) <= m0)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Wait that ignores the abort flag (tear-down): bounded by `limit_ns`.
FP8FG_DEV bool wait_plain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;   // no timer read on the fast path
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

FP8FG_DEV uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------ producer ---
// One thread: the A and B operand tiles of every chunk, by TMA.
template <int kRowB>
FP8FG_DEV void run_producer(Smem<kRowB>& sm, const CUtensorMap* tmap_a, const CUtensorMap* tmap_b, const Params& p,
                            int64_t m_tiles, int64_t n_tiles, int64_t kb) {
    constexpr int ST = Smem<kRowB>::kStages;
    volatile int* abort_flag = &sm.abort_flag;
    uint32_t g_ab = 0;  // chunks whose operand copies were issued
    const int64_t num_tiles = m_tiles * n_tiles;
    bool ok = true;
    for (int64_t t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int64_t m0, n0;
        tile_origin(t, m_tiles, n_tiles, p.m_fastest, m0, n0);
        const int e = p.offsets ? expert_of(p.offsets, p.G, m0) : 0;
        for (int64_t c = 0; c < kb; ++c) {
            const uint32_t s = g_ab % ST;
            if (g_ab >= static_cast<uint32_t>(ST)) {
                // Stage s is free once the load of chunk d = g_ab - ST into it
                // has landed and that chunk's MMAs have completed.  The first
                // wait is needed on the abort path only: a chunk whose
                // operands the watcher did not confirm is committed without
                // MMAs, possibly while its load is still in flight, and a
                // second load into the stage must never be issued on top of
                // it (each stage has at most one load in flight, so the
                // tear-down below can wait for every copy to land).
                const uint32_t d = g_ab - ST;
                if (!mbar_wait_bounded(smem_u32(&sm.full[s]), (d / ST) & 1, abort_flag, p.status, p.limit_ns,
                                       kErrTimeout) ||
                    !mbar_wait_bounded(smem_u32(&sm.done[d % kDone]), (d / kDone) & 1, abort_flag, p.status,
                                       p.limit_ns, kErrTimeout)) {
                    ok = false;
                    break;
                }
            }
            const uint32_t fb = smem_u32(&sm.full[s]);
            mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
            tma_load_2d(smem_u32(sm.a[s]), tmap_a, static_cast<int32_t>(c * BK), static_cast<int32_t>(m0), fb);
            if (p.offsets)
                tma_load_3d(smem_u32(sm.b[s]), tmap_b, static_cast<int32_t>(c * BK), static_cast<int32_t>(n0), e, fb);
            else
                tma_load_2d(smem_u32(sm.b[s]), tmap_b, static_cast<int32_t>(c * BK), static_cast<int32_t>(n0), fb);
            ++g_ab;
        }
    }
    if (!ok) {
        // abort: let the copies already issued land before the CTA exits; a
        // copy still in flight after the limit is recorded as a tear-down
        // failure (the CTA's shared memory is released with it pending)
        bool landed = true;
        for (uint32_t s = 0; s < ST && s < g_ab; ++s) {
            const uint32_t last = s + ST * ((g_ab - 1 - s) / ST);
            landed &= wait_plain(smem_u32(&sm.full[s]), (last / ST) & 1, kTeardownLimitNs);
        }
        if (!landed) atomicExch(p.status, kErrTeardown);
    }
}

// ---------------------------------------------- per-row scale stager ---
// Per-row B scales only; warp 3.  The ring's slots hold kScaleGroup chunks
// each.  For every group of chunks, in the MMA warp's order: wait until the
// promotion warps have released the slot, then copy each chunk's B scales
// of the tile's 256 columns and A scales of its 128 rows from global memory
// straight into the slot by cp.async, permuted so that a promotion thread
// (run_epilogue_rowb) finds its 4 A scales in one 16-byte run and the B
// scales of each 32 of its columns in two.  Every lane then makes the
// slot's "full" barrier (count 32) take its arrival once its own copies have
// landed, so the warp neither holds the scales in registers nor waits for
// the loads.  Layouts of a chunk in a slot:
//   B: position 128 h + 32 s + 16 p + 4 q + 2 b + e holds column
//      128 h + 32 s + 8 (2 p + b) + 2 q + e of the tile;
//   A: position 32 u + 4 r + k holds row 32 u + r + 8 k.
// Lane l fills positions 4 l .. 4 l + 3 of A and of each half h of B.  The
// scales are not copied by TMA because the permutation has 8-byte
// granularity; doing it here keeps the promotion warps' shared loads (which
// compete with the tensor core's operand reads) at 9 per chunk instead of
// 20, and one slot per group keeps their ring handshakes at one per group.
FP8FG_DEV void run_scales(Smem<1>& sm, const Params& p, int64_t m_tiles, int64_t n_tiles, int64_t kb, int lane) {
    constexpr int SL = Smem<1>::kSlots, G = kScaleGroup;
    volatile int* abort_flag = &sm.abort_flag;
    const int64_t num_tiles = m_tiles * n_tiles;
    // this lane's B columns cb, cb + 1, cb + 8, cb + 9 (and + 128), A rows ra + 8 k
    const int cb = 32 * (lane >> 3) + 16 * ((lane >> 2) & 1) + 2 * (lane & 3);
    const int ra = 32 * (lane >> 3) + (lane & 7);
    uint32_t gq = 0;   // groups of G chunks staged
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int64_t m0, n0;
        tile_origin(t, m_tiles, n_tiles, p.m_fastest, m0, n0);
        const bool hi = n0 + 128 < p.N;   // the tile's second 128 columns exist (N is a multiple of 128)
        for (int64_t c0 = 0; c0 < kb; c0 += G, ++gq) {
            const uint32_t sl = gq % SL, sph = (gq / SL) & 1;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_bounded(smem_u32(&sm.sempty[sl]), sph ^ 1, abort_flag, p.status, p.limit_ns,
                                       kErrTimeout);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                cp_async_wait_all();   // no copy of this warp outlives it
                return;
            }
            // the group's scales go straight from global memory into their
            // permuted places by cp.async (no registers held, no wait here);
            // the slot's "full" barrier counts this lane's arrival once its
            // copies have landed.  Columns past N and chunks past the tile's
            // last are not copied (never read).
#pragma unroll
            for (int q = 0; q < G; ++q) {
                const int64_t c = c0 + q;
                if (c < kb) {
                    const float* sbr = p.sb + c * p.N + n0 + cb;
                    const float* sar = p.sa + c * p.M + m0 + ra;
                    const uint32_t sb_s = smem_u32(sm.sb[sl][q]) + 16 * lane, sa_s = smem_u32(sm.sa[sl][q]) + 16 * lane;
                    cp_async_8(sb_s, sbr);
                    cp_async_8(sb_s + 8, sbr + 8);
                    if (hi) {
                        cp_async_8(sb_s + 512, sbr + 128);
                        cp_async_8(sb_s + 520, sbr + 136);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) cp_async_4(sa_s + 4 * k, sar + 8 * k);
                }
            }
            cp_async_mbar_arrive_noinc(smem_u32(&sm.sfull[sl]));
        }
    }
    cp_async_wait_all();
}

// ------------------------------------------------------- operand watcher ---
// Whole warp; lane 0 waits.  For every chunk, in the MMA warp's order, wait
// for the stage's "full" mbarrier (skipped after a failed wait) and meet the
// MMA warp on kOpsBar, passing whether this or an earlier wait failed.  Both
// warps meet exactly once per chunk on every path, so neither runs ahead.
template <int kRowB>
FP8FG_DEV void run_watch(Smem<kRowB>& sm, const Params& p, int64_t m_tiles, int64_t n_tiles, int64_t kb, int lane) {
    constexpr int ST = Smem<kRowB>::kStages;
    volatile int* abort_flag = &sm.abort_flag;
    uint32_t g = 0;
    const int64_t num_tiles = m_tiles * n_tiles;
    bool ok = true;   // warp-uniform
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        for (int64_t c = 0; c < kb; ++c, ++g) {
            const uint32_t s = g % ST, ph = (g / ST) & 1;
            if (ok) {
                bool f = true;
                if (lane == 0)
                    f = mbar_wait_bounded(smem_u32(&sm.full[s]), ph, abort_flag, p.status, p.limit_ns, kErrTimeout);
                ok = __shfl_sync(0xffffffffu, f, 0) != 0;
            }
            named_sync_or<kOpsThreads>(kOpsBar, !ok);
        }
    }
}

// ----------------------------------------------------------------- MMA ---
// Whole warp; lane 0 issues.  Lock step with the promotion warps: before
// chunk g (g >= 2) the warp takes the hand-back of chunk g-2 on the named
// barrier of its buffer, and for every chunk, aborted or not, lane 0 commits
// the chunk's "done" mbarrier (with no MMA after an abort the commit only
// tracks the earlier ones).  A promotion warp arrives for chunk g only after
// that commit, so no arrival can run ahead of the MMA warp's bar.sync, and
// every bar.sync is matched by the 8 arrivals of a chunk already committed.
// The chunk's operands are reported by the watcher on kOpsBar, before any
// MMA of the chunk is issued.  The chunks of all the CTA's tiles form one
// flat loop with the stage, buffer and descriptors stepped incrementally.
template <int kRowB>
FP8FG_DEV void run_mma(Smem<kRowB>& sm, uint32_t tmem_base, const Params& p, int64_t m_tiles, int64_t n_tiles,
                       int64_t kb, int lane) {
    constexpr int ST = Smem<kRowB>::kStages;
    const int64_t num_tiles = m_tiles * n_tiles;
    const int64_t b = blockIdx.x;
    const uint32_t chunks = b < num_tiles ? static_cast<uint32_t>(((num_tiles - 1 - b) / gridDim.x + 1) * kb) : 0u;
    // descriptors of stage 0; stage s is A_BYTES * s (B_BYTES * s) further,
    // i.e. (A_BYTES >> 4) * s in the descriptor's start-address field
    const uint64_t adesc0 = smem_desc_sw128(smem_u32(sm.a[0]));
    const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sm.b[0]));
    uint32_t soff_a = 0, soff_b = 0, s = 0, buf = 0;
    bool ok = true;   // warp-uniform
    for (uint32_t g = 0; g < chunks; ++g) {
        if (g >= NBUF) named_sync<kRelThreads>(1 + static_cast<int>(buf));
        if (named_sync_or<kOpsThreads>(kOpsBar, false)) ok = false;
        if (lane == 0) {
            if (ok) {
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                const uint64_t adesc = adesc0 + soff_a, bdesc = bdesc0 + soff_b;
#pragma unroll
                for (int kk = 0; kk < BK / MMA_K; ++kk) {
                    // advance 32 bytes along K inside the 128-byte swizzle atom
                    const uint64_t koff = static_cast<uint64_t>((kk * MMA_K) >> 4);
                    mma_f8f6f4(d_tmem, adesc + koff, bdesc + koff, kIdesc, kk > 0 ? 1u : 0u);
                }
            }
            mma_commit(smem_u32(&sm.done[g & (kDone - 1)]));
        }
        __syncwarp();
        buf ^= 1u;
        if (++s == static_cast<uint32_t>(ST)) {
            s = 0;
            soff_a = 0;
            soff_b = 0;
        } else {
            soff_a += A_BYTES >> 4;
            soff_b += B_BYTES >> 4;
        }
    }
    // the last hand-back of each buffer that was used
    for (uint32_t bb = 0; bb < NBUF; ++bb)
        if (chunks > bb) named_sync<kRelThreads>(1 + static_cast<int>(bb));
    if (lane == 0) {
        // every MMA issued by this thread has finished before TMEM is released
        mma_commit(smem_u32(&sm.drain));
        if (!wait_plain(smem_u32(&sm.drain), 0, 10 * kTeardownLimitNs)) atomicExch(p.status, kErrTeardown);
    }
    __syncwarp();
}

// ------------------------------------------------------------ promotion ---
// acc[0..15] += P[0..15] * scale (block B scales: one scale per thread and chunk).
FP8FG_DEV void promote16(float* acc, const uint32_t (&r)[16], float scale) {
#pragma unroll
    for (int k = 0; k < 16; k += 2)
        fma2(acc[k], acc[k + 1], __uint_as_float(r[k]), __uint_as_float(r[k + 1]), scale, scale);
}

// A tile's origin and the first scales its promotion needs, loaded one tile
// ahead (while the previous tile's outputs are being stored) so that the
// first chunk of a tile does not wait for them.
struct TileScales {
    int64_t m0, col0;
    bool active;
    const float* sbp;       // block B scales of this warp's 128 columns, chunk 0
    const float* sap;       // A scale of this thread's row, chunk 0
    float sb_cur, sb_nxt;   // block B scales of chunks 32 w + l (lane l): the current window w, the next
    float q[4];             // A scales of chunks 0 .. 3 (a chunk past the tile's last repeats the last)
};

FP8FG_DEV TileScales load_tile_scales(int64_t t, const Params& p, int64_t m_tiles, int64_t n_tiles, int64_t kb,
                                      int half, int row, int lane) {
    TileScales ts;
    int64_t n0;
    tile_origin(t, m_tiles, n_tiles, p.m_fastest, ts.m0, n0);
    ts.col0 = n0 + ECOLS * half;
    ts.active = ts.col0 < p.N;
    ts.sb_cur = 0.0f;
    ts.sb_nxt = 0.0f;
    const int e = p.offsets ? expert_of(p.offsets, p.G, ts.m0) : 0;
    ts.sbp = p.sb + e * p.sb_group_stride + (ts.col0 / 128) * p.sb_stride_n;
    if (ts.active && lane < kb) ts.sb_cur = __ldg(ts.sbp + lane * p.sb_stride_k);
    if (ts.active && lane + 32 < kb) ts.sb_nxt = __ldg(ts.sbp + (lane + 32) * p.sb_stride_k);
    // rows past M (a partial last row tile) read row M - 1's scales: their
    // partial sums are zero (the A box reads zeros there) and never stored
    ts.sap = p.sa + min(ts.m0 + row, p.M - 1);
    // (indices clamped to the last chunk instead of a select on the loaded
    // value: a select would make the thread wait for the load to return)
#pragma unroll
    for (int j = 0; j < 4; ++j) ts.q[j] = __ldg(ts.sap + min(static_cast<int64_t>(j), kb - 1) * p.M);
    return ts;
}

FP8FG_DEV void run_epilogue(Smem<0>& sm, uint32_t tmem_base, const Params& p, const CUtensorMap* tmap_d,
                            int64_t m_tiles, int64_t n_tiles, int64_t kb, int warp, int lane) {
    volatile int* abort_flag = &sm.abort_flag;
    const int quad = warp & 3;          // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int half = (warp - 4) >> 2;   // columns ECOLS*half .. ECOLS*half+ECOLS-1 of the tile
    const int row = quad * 32 + lane;   // tile row owned by this thread
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t ob = smem_u32(sm.out[warp - 4]);
    const int64_t num_tiles = m_tiles * n_tiles;
    uint32_t g = 0;
    bool dead = false;   // after a failed wait: no work, but still one hand-back per chunk
    bool timed_out = false;
    TileScales nts = load_tile_scales(blockIdx.x, p, m_tiles, n_tiles, kb, half, row, lane);
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        const int64_t m0 = nts.m0, col0 = nts.col0;
        const bool active = nts.active;
        const float* sbp = nts.sbp;
        const float* sap = nts.sap;
        float sb_cur = nts.sb_cur, sb_nxt = nts.sb_nxt;
        // A scales of four consecutive chunks in a register ring: the chunk
        // loop below is unrolled by four and each copy of its body names its
        // own ring register, so the scale of chunk c + 4, loaded while chunk
        // c is promoted, is first read four chunks later (a rotation of the
        // registers would read the newest load at once and wait for it)
        float qa0 = nts.q[0], qa1 = nts.q[1], qa2 = nts.q[2], qa3 = nts.q[3];
        float acc[ECOLS];
#pragma unroll
        for (int j = 0; j < ECOLS; ++j) acc[j] = 0.0f;
        auto chunk = [&](int64_t c, float& qa) {
            const uint32_t buf = g % NBUF;
            if (c > 0 && (c & 31) == 0) {
                sb_cur = sb_nxt;
                if (active) sb_nxt = __ldg(sbp + min(c + 32 + lane, kb - 1) * p.sb_stride_k);
            }
            const float sa_i = qa;
            // chunk c + 4's scale; past the tile's last chunk the (unused)
            // load repeats the last one: an unconditional load
            qa = __ldg(sap + min(c + 4, kb - 1) * p.M);
            // Every lane waits (each gets the barrier's acquire).  The MMA
            // warp commits this barrier for every chunk, aborted or not, so
            // the wait ignores the abort flag; its limit is far above the
            // longest wait the commit can depend on.
            // (After such a wait has failed, which the lock step rules out,
            // the later ones are kept short so the kernel still ends.)
            bool ok = wait_plain(smem_u32(&sm.done[g & (kDone - 1)]), (g / kDone) & 1,
                                 timed_out ? 1000000ull : kHandoffLimitNs);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    atomicCAS(p.status, 0, kErrTimeout);
                    *abort_flag = 1;
                }
                dead = true;
                timed_out = true;
            }
            tc_fence_after();
            const float sbv = __shfl_sync(0xffffffffu, sb_cur, static_cast<int>(c & 31));
            if (active && !dead) {
                const uint32_t taddr = tmem_base + t_lane + buf * BN + ECOLS * half;
                const float scale = sa_i * sbv;
                // ECOLS / 16 loads of 16 columns; the next load is in flight
                // while the previous 16 columns are folded in (16, not 32:
                // with 32 the registers spilled)
                constexpr int NJ = ECOLS / 16;
                uint32_t r[2][16];
                tmem_ld_32x32b_x16(taddr, r[0]);
                tmem_ld_wait(r[0]);
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    if (j + 1 < NJ) tmem_ld_32x32b_x16(taddr + 16 * (j + 1), r[(j + 1) & 1]);
                    promote16(acc + 16 * j, r[j & 1], scale);
                    if (j + 1 < NJ) tmem_ld_wait(r[(j + 1) & 1]);
                }
            }
            // the buffer goes back only after the loaded registers are consumed
            tc_fence_before();
            named_arrive<kRelThreads>(1 + static_cast<int>(buf));
            ++g;
        };
        for (int64_t c = 0; c < kb; c += 4) {
            chunk(c, qa0);
            if (c + 1 < kb) chunk(c + 1, qa1);
            if (c + 2 < kb) chunk(c + 2, qa2);
            if (c + 3 < kb) chunk(c + 3, qa3);
        }
        if (t + gridDim.x < num_tiles)
            nts = load_tile_scales(t + gridDim.x, p, m_tiles, n_tiles, kb, half, row, lane);
        // (a warp whose 32 rows all lie past M, in a partial last row tile,
        // stores nothing; a store box that crosses M is clipped by TMA)
        if (!active || dead || m0 + quad * 32 >= p.M) continue;
        // 32 rows x 128 columns of this warp -> shared memory (row = lane,
        // 16-byte chunk k of each 128-byte row at k ^ (row & 7): the 128-byte
        // swizzle of the output map) -> one TMA store per 128 bytes of row;
        // before the buffer is rewritten the previous store must have read it.
        // (A second staging buffer per warp was slower: above 196 KB of
        // shared memory the L1 left for the scale loads shrinks to 28 KB.)
        const int32_t gy = static_cast<int32_t>(m0 + quad * 32);
        constexpr int kRounds = ECOLS / 32;   // FP32 rounds; BF16 needs half as many
        const int rounds = p.out_bf16 ? kRounds / 2 : kRounds;
#pragma unroll
        for (int rd = 0; rd < kRounds; ++rd) {
            if (rd < rounds) {
                const uint32_t orow = ob + static_cast<uint32_t>(lane) * 128;
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
                if (p.out_bf16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float* a8 = acc + (64 * rd) % ECOLS + 8 * k;   // rd < kRounds / 2 here
                        st_shared_v4(orow + ((k ^ (lane & 7)) << 4), pack_bf16x2(a8[0], a8[1]),
                                     pack_bf16x2(a8[2], a8[3]), pack_bf16x2(a8[4], a8[5]), pack_bf16x2(a8[6], a8[7]));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float* a4 = acc + 32 * rd + 4 * k;
                        st_shared_v4(orow + ((k ^ (lane & 7)) << 4), __float_as_uint(a4[0]), __float_as_uint(a4[1]),
                                     __float_as_uint(a4[2]), __float_as_uint(a4[3]));
                    }
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmap_d, ob, static_cast<int32_t>(col0 + (p.out_bf16 ? 64 : 32) * rd), gy);
                    bulk_commit_group();
                }
            }
        }
    }
    if (lane == 0) bulk_wait_group0();   // every store of this warp has completed
    __syncwarp();
}

// ---------------------------------------- promotion, per-row B scales ---
// Per-row B scales (Wgrad: both operands scaled per 128-token chunk, one
// scale per output row i and one per output column j): every partial sum
// takes its own product sa_i * sb_j, two FP32 operations per sum.  The
// chunk's B and A scales come from the shared ring warp 3 fills in a
// permuted order (run_scales).  TMEM is read with the 16x256b shape, so that a
// thread holds 4 rows x 32 columns of its warp's 32 x 128 block and needs 32
// B scales and 4 A scales per chunk: a thread that held one whole row would
// need all 128 of its columns' B scales every chunk.  Shared-memory loads
// compete with the tensor core, which streams its operands from shared
// memory (each load wavefront delays the MMAs), so their number matters
// more than their latency.
//
// Thread (g = lane / 4, q = lane % 4) of promotion warp (quad, half):
//   rows    32 quad + 16 rh + 8 rr + g          (rh, rr in {0, 1})
//   columns ECOLS half + 8 b + 2 q + e          (b < 16, e in {0, 1})
// TMEM load j (0..7) reads the 16 rows of rh = j % 2 and the column blocks
// b = 4 (j / 2) + bb (bb < 4); its register 4 bb + 2 rr + e is folded into
// acc[16 j + 4 bb + 2 rr + e].
FP8FG_DEV void run_epilogue_rowb(Smem<1>& sm, uint32_t tmem_base, const Params& p, const CUtensorMap* tmap_d,
                                 int64_t m_tiles, int64_t n_tiles, int64_t kb, int warp, int lane) {
    constexpr int SL = Smem<1>::kSlots, G = kScaleGroup;
    volatile int* abort_flag = &sm.abort_flag;
    const int quad = warp & 3;          // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int half = (warp - 4) >> 2;   // columns ECOLS*half .. ECOLS*half+ECOLS-1 of the tile
    const int g4 = lane >> 2, q = lane & 3;
    const uint32_t ob = smem_u32(sm.out[warp - 4]);
    const int64_t num_tiles = m_tiles * n_tiles;
    uint32_t g = 0;
    uint32_t gq = 0;   // scale groups (kScaleGroup chunks, one ring slot each) consumed
    bool dead = false;   // after a failed wait: no work, but still one hand-back per chunk
    bool timed_out = false;
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int64_t m0, n0;
        tile_origin(t, m_tiles, n_tiles, p.m_fastest, m0, n0);
        const int64_t col0 = n0 + ECOLS * half;
        const bool active = col0 < p.N;
        float acc[ECOLS];
#pragma unroll
        for (int j = 0; j < ECOLS; ++j) acc[j] = 0.0f;
        for (int64_t c = 0; c < kb; ++c) {
            const uint32_t buf = g % NBUF;
            const uint32_t sl = gq % SL, sph = (gq / SL) & 1;
            const int cq = static_cast<int>(c % G);   // chunk within the slot's group
            // (the waits as in run_epilogue)
            bool ok = wait_plain(smem_u32(&sm.done[g & (kDone - 1)]), (g / kDone) & 1,
                                 timed_out ? 1000000ull : kHandoffLimitNs);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    atomicCAS(p.status, 0, kErrTimeout);
                    *abort_flag = 1;
                }
                dead = true;
                timed_out = true;
            }
            if (!dead && cq == 0) {   // the group's scales have been staged
                ok = mbar_wait_bounded(smem_u32(&sm.sfull[sl]), sph, abort_flag, p.status, p.limit_ns, kErrTimeout);
                if (!__all_sync(0xffffffffu, ok)) dead = true;
            }
            tc_fence_after();
            if (active && !dead) {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * BN + ECOLS * half;
                // the slot's permuted layouts (run_scales): A rows 8k + g4 of
                // this warp's 32 at 4 g4 + k, B columns 8 bb + 2 q + e of each
                // 32 at 16 (bb / 2) + 4 q + 2 (bb % 2) + e
                const uint32_t sbp = smem_u32(sm.sb[sl][cq] + ECOLS * half + 4 * q);
                const uint4 sa4 = ld_shared_v4(smem_u32(sm.sa[sl][cq] + quad * 32 + 4 * g4));
                // A scales of rows 8k + g4: (rh, rr) = (k / 2, k % 2)
                const float sav[4] = {__uint_as_float(sa4.x), __uint_as_float(sa4.y), __uint_as_float(sa4.z),
                                      __uint_as_float(sa4.w)};
                float2 sbv[4];  // B scales of the current 32 columns
                auto load_sb = [&](int seg) {
                    const uint4 lo = ld_shared_v4(sbp + 128 * seg), hi = ld_shared_v4(sbp + 128 * seg + 64);
                    sbv[0] = make_float2(__uint_as_float(lo.x), __uint_as_float(lo.y));
                    sbv[1] = make_float2(__uint_as_float(lo.z), __uint_as_float(lo.w));
                    sbv[2] = make_float2(__uint_as_float(hi.x), __uint_as_float(hi.y));
                    sbv[3] = make_float2(__uint_as_float(hi.z), __uint_as_float(hi.w));
                };
                load_sb(0);
                uint32_t r[2][16];
                tmem_ld_16x256b_x4(taddr, r[0]);
                tmem_ld_wait(r[0]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j + 1 < 8)
                        tmem_ld_16x256b_x4(taddr + (static_cast<uint32_t>(16 * ((j + 1) & 1)) << 16) +
                                               32 * ((j + 1) >> 1),
                                           r[(j + 1) & 1]);
                    const int rh = j & 1;
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            float x0 = __uint_as_float(r[j & 1][4 * bb + 2 * rr]);
                            float x1 = __uint_as_float(r[j & 1][4 * bb + 2 * rr + 1]);
                            mul2(x0, x1, sbv[bb].x, sbv[bb].y);
                            const float sa_r = sav[2 * rh + rr];
                            float* a2 = acc + 16 * j + 4 * bb + 2 * rr;
                            fma2(a2[0], a2[1], x0, x1, sa_r, sa_r);
                        }
                    }
                    if (j + 1 < 8) {
                        if (j & 1) load_sb((j + 1) >> 1);   // the next load starts the next 32 columns
                        tmem_ld_wait(r[(j + 1) & 1]);
                    }
                }
            }
            // the buffer goes back only after the loaded registers are consumed
            tc_fence_before();
            named_arrive<kRelThreads>(1 + static_cast<int>(buf));
            if (cq == G - 1 || c == kb - 1) {   // the group's last chunk: the slot goes back
                __syncwarp();   // every lane's scale loads from the slot are done
                if (!dead && lane == 0) mbar_arrive(smem_u32(&sm.sempty[sl]));
                ++gq;
            }
            ++g;
        }
        if (!active || dead) continue;
        // 32 rows x 128 columns of this warp -> the warp's staging buffer
        // (row-major 128-byte rows, 16-byte chunk k of row r at k ^ (r & 7):
        // the output map's 128-byte swizzle) -> one TMA store per 128 bytes
        // of row, as in run_epilogue, from this thread's 4 rows x 32 columns.
        const int32_t gy = static_cast<int32_t>(m0 + quad * 32);
        if (p.out_bf16) {
#pragma unroll
            for (int rd = 0; rd < 2; ++rd) {   // 64 columns per round: blocks b = 8 rd + bp
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
#pragma unroll
                for (int bp = 0; bp < 8; ++bp) {
                    const int b = 8 * rd + bp;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rh = k >> 1, rr = k & 1, row = 16 * rh + 8 * rr + g4;
                        const float* a2 = acc + 16 * (2 * (b >> 2) + rh) + 4 * (b & 3) + 2 * rr;
                        st_shared_u32(ob + static_cast<uint32_t>(row) * 128 + ((bp ^ (row & 7)) << 4) + 4 * q,
                                      pack_bf16x2(a2[0], a2[1]));
                    }
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmap_d, ob, static_cast<int32_t>(col0 + 64 * rd), gy);
                    bulk_commit_group();
                }
            }
        } else {
#pragma unroll
            for (int rd = 0; rd < 4; ++rd) {   // 32 columns per round: blocks b = 4 rd + bb
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int kc = 2 * bb + (q >> 1);   // 16-byte chunk of the row
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rh = k >> 1, rr = k & 1, row = 16 * rh + 8 * rr + g4;
                        const float* a2 = acc + 16 * (2 * rd + rh) + 4 * bb + 2 * rr;
                        st_shared_v2(ob + static_cast<uint32_t>(row) * 128 + ((kc ^ (row & 7)) << 4) + 8 * (q & 1),
                                     __float_as_uint(a2[0]), __float_as_uint(a2[1]));
                    }
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmap_d, ob, static_cast<int32_t>(col0 + 32 * rd), gy);
                    bulk_commit_group();
                }
            }
        }
    }
    if (lane == 0) bulk_wait_group0();   // every store of this warp has completed
    __syncwarp();
}

// ------------------------------------------------ fused A quantization ---
// Phase 1 of fp8_gemm_quant_a: this CTA's share of the 1x128 quantization of
// the BF16 A operand into q_a / s_a, the buffers the GEMM phase then reads
// (the codes through the A tensor map).  Work: 128-row x 128-column tiles in
// band-major order (tile t: 128-row band t / kb, group column t % kb), tile t
// done by CTA t % gridDim.x.  Thread 0 streams the CTA's tiles with TMA (two
// 128-row x 64-column boxes per tile, 128-byte swizzle) into a ring of five
// 32 KB slots laid over the GEMM's idle operand stages and output staging; the 256 threads of
// warps 4-11 quantize each tile from shared memory with
// fp8_quant_act_1x128's mapping and arithmetic (a lane quad per row group,
// lane j holding chunks 2j, 2j+1, 2j+8, 2j+9, written as two 16-byte runs;
// two rows per thread), so the codes
// and scales are the ones that quantizer writes; once the CTA's share is
// done, each of its tiles is added to its band's counter with a release at
// GPU scope.  Sources: DeepSeek-V3 FP8 post
// (innerforce.co.kr), fine-grained quantization paragraph (1x128 tiles,
// max-abs scaling, online) and low-precision storage paragraph (activations
// kept in FP8).
constexpr int kPhase1Bar = 4;          // named barrier of the 256 phase-1 threads
constexpr int kPhase1Threads = 256;
constexpr int kP1Slots = 5;
constexpr uint32_t kP1SlotBytes = 128 * 128 * 2;   // one BF16 tile: two 16 KB boxes
constexpr uint32_t kP1BoxBytes = kP1SlotBytes / 2;

template <int kRowB>
FP8FG_DEV uint32_t p1_slot(Smem<kRowB>& sm, uint32_t i) {
    static_assert(sizeof(sm.a) + sizeof(sm.b) + sizeof(sm.out) >= kP1Slots * kP1SlotBytes,
                  "phase-1 ring inside the operand stages and the output staging buffers");
    return smem_u32(&sm.a[0][0]) + (i % kP1Slots) * kP1SlotBytes;
}

// Thread 0: load the CTA's tiles into the ring.  Returns the number of tiles
// whose loads were issued (all of them unless a wait ran out).
template <int kRowB>
FP8FG_DEV uint32_t p1_load(Smem<kRowB>& sm, const CUtensorMap* tmap_x, const Params& p, int64_t units, int64_t kb) {
    volatile int* abort_flag = &sm.abort_flag;
    uint32_t i = 0;
    for (int64_t t = blockIdx.x; t < units; t += gridDim.x, ++i) {
        if (i >= kP1Slots) {
            const uint32_t prev = i - kP1Slots;   // the tile that used this slot
            if (!mbar_wait_bounded(smem_u32(&sm.pempty[prev % kP1Slots]), (prev / kP1Slots) & 1, abort_flag,
                                   p.status, p.limit_ns, kErrTimeout))
                break;
        }
        const uint32_t m = static_cast<uint32_t>(t) / static_cast<uint32_t>(kb);
        const uint32_t c = static_cast<uint32_t>(t) - m * static_cast<uint32_t>(kb);
        const uint32_t fb = smem_u32(&sm.pfull[i % kP1Slots]), dst = p1_slot(sm, i);
        mbar_arrive_expect_tx(fb, kP1SlotBytes);
        tma_load_2d(dst, tmap_x, static_cast<int32_t>(c * BK), static_cast<int32_t>(m * BM), fb);
        tma_load_2d(dst + kP1BoxBytes, tmap_x, static_cast<int32_t>(c * BK + 64), static_cast<int32_t>(m * BM), fb);
    }
    return i;
}

// Warps 4-11: quantize the CTA's tiles from the ring.  Returns false after a
// failed wait (the kernel then computes nothing).
template <int kRowB>
FP8FG_DEV bool p1_quantize(Smem<kRowB>& sm, const Params& p, int64_t units, int64_t kb, int tid) {
    volatile int* abort_flag = &sm.abort_flag;
    const int j = tid & 3;     // chunks 2j, 2j+1, 2j+8, 2j+9 of the row group
    const int rq = tid >> 2;   // row within a 64-row half of the tile
    const int lane = tid & 31;
    bool ok = true;            // warp-uniform
    uint32_t i = 0;
    for (int64_t t = blockIdx.x; t < units; t += gridDim.x, ++i) {
        if (ok) {
            bool f = mbar_wait_bounded(smem_u32(&sm.pfull[i % kP1Slots]), (i / kP1Slots) & 1, abort_flag, p.status,
                                       p.limit_ns, kErrTimeout);
            ok = __all_sync(0xffffffffu, f);
        }
        if (ok) {
            // 32-bit index arithmetic: the tile count is below 2^31 (checked on the host)
            const uint32_t m = static_cast<uint32_t>(t) / static_cast<uint32_t>(kb);
            const uint32_t c = static_cast<uint32_t>(t) - m * static_cast<uint32_t>(kb);
            const uint32_t slot = p1_slot(sm, i);
            // both rows' chunks first (eight loads in flight), then the groups
            uint4 v[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = rq + 64 * u;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // chunk 2j + (k & 1) + 8 (k / 2) of the row: box k / 2, 16-byte unit
                    // 2j + (k & 1) of its 128-byte row, 128-byte swizzle (the two rows of
                    // a quarter-warp then read disjoint banks)
                    const uint32_t unit = static_cast<uint32_t>(2 * j + (k & 1)) ^ static_cast<uint32_t>(r & 7);
                    v[u][k] = ld_shared_v4(slot + (k >> 1) * kP1BoxBytes + r * 128 + (unit << 4));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = rq + 64 * u;
                const float amax = quad_amax_bf16(v[u]);
                const float s = __fdiv_rn(amax, 448.0f);
                const GroupScale gs(s);
                const int64_t row = static_cast<int64_t>(m) * BM + r;
                // codes of chunks 2j, 2j+1 and of chunks 2j+8, 2j+9: two 16-byte stores
                uint4* dst = reinterpret_cast<uint4*>(p.qa) + (row * p.K + static_cast<int64_t>(c) * BK) / 16 + j;
                with_mode(gs, [&](auto md) {
                    constexpr int kM = decltype(md)::value;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 out;
                        out.x = quant_quad_bf16<kM>(v[u][2 * h].x, v[u][2 * h].y, gs);
                        out.y = quant_quad_bf16<kM>(v[u][2 * h].z, v[u][2 * h].w, gs);
                        out.z = quant_quad_bf16<kM>(v[u][2 * h + 1].x, v[u][2 * h + 1].y, gs);
                        out.w = quant_quad_bf16<kM>(v[u][2 * h + 1].z, v[u][2 * h + 1].w, gs);
                        __stcs(dst + 4 * h, out);
                    }
                });
                if (j == 0) p.sa_out[static_cast<int64_t>(c) * p.M + row] = s;
            }
        }
        // the slot goes back to the loader (its reads are ordered before the
        // next TMA write by the mbarrier, as in any TMA consumer ring)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.pempty[i % kP1Slots]));
    }
    // Publish the CTA's tiles once, at the end (fences per tile measured a
    // store round trip each): this thread's shared reads before the GEMM's
    // TMA rewrites the stages and its global writes before later TMA reads
    // of them; the 256 threads' writes; then one GPU-scope fence and a
    // relaxed add per tile to its band's counter.
    fence_proxy_async_shared();
    fence_proxy_async_global();
    named_sync<kPhase1Threads>(kPhase1Bar);
    if (tid == 0 && ok) {
        __threadfence();
        for (int64_t t = blockIdx.x; t < units; t += gridDim.x) atomicAdd(p.band_flags + t / kb, 1);
    }
    return ok;
}

// Warp 0 of every CTA: wait until every band's kb tiles are published
// (acquire), lane l polling bands l, l + 32, ... (in parallel: one polling
// thread reading the counters one after another took several microseconds
// more), each lane bounded by the wait limit.  Returns the same result in
// every lane; a timeout records FP8FG_ERR_TIMEOUT and the CTA computes
// nothing.
FP8FG_DEV bool wait_bands(const Params& p, int64_t m_tiles, int64_t kb, int lane) {
    const uint64_t t0 = globaltimer_ns();
    bool ok = true;
    for (int64_t m = lane; ok && m < m_tiles; m += 32) {
        while (ld_acquire_gpu(p.band_flags + m) < kb) {
            if (globaltimer_ns() - t0 > p.limit_ns) {
                ok = false;
                break;
            }
        }
    }
    __syncwarp();   // every lane's acquires before lane 0's TMA reads of q_a
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) {
        if (!ok) atomicCAS(p.status, 0, kErrTimeout);
        fence_proxy_async_global();   // before this thread (the producer) issues TMA reads of q_a
    }
    return ok;
}

template <int kRowB, bool kFusedA>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                            const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_x,
                            const Params p) {
    using S = Smem<kRowB>;
    extern __shared__ uint8_t smem_raw[];
    S& sm = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m_tiles = p.m_tiles, n_tiles = (p.N + BN - 1) / BN, kb = p.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) mbar_init(smem_u32(&sm.full[s]), 1);
        for (uint32_t d = 0; d < kDone; ++d) mbar_init(smem_u32(&sm.done[d]), 1);
        for (int s = 0; s < S::kSlots; ++s) {
            mbar_init(smem_u32(&sm.sfull[s]), 32);   // the 32 lanes of the scale stager
            mbar_init(smem_u32(&sm.sempty[s]), EPI_WARPS);
        }
        mbar_init(smem_u32(&sm.drain), 1);
        for (int s = 0; s < kP1Slots; ++s) {
            mbar_init(smem_u32(&sm.pfull[s]), 1);
            mbar_init(smem_u32(&sm.pempty[s]), EPI_WARPS);
        }
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (kFusedA && threadIdx.x == 0) prefetch_tensormap(&tmap_x);
    if (kFusedA) __syncthreads();   // the ring's barriers are initialised before phase 1 uses them
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_d);
    }
    if (warp == 1) tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
    int bad = 0;
    if (p.offsets) {
        // grouped offsets must start at 0, end at M, be non-decreasing and
        // multiples of 128; otherwise nothing is computed or written
        for (int g = threadIdx.x; g <= p.G; g += THREADS) {
            const int64_t o = __ldg(p.offsets + g);
            if (o < 0 || o > p.M || (o % BM) != 0) bad = 1;
            if (g == 0 && o != 0) bad = 1;
            if (g == p.G && o != p.M) bad = 1;
            if (g > 0 && static_cast<int64_t>(__ldg(p.offsets + g - 1)) > o) bad = 1;
        }
    }
    int stop = 0;
    if (kFusedA) {
        // phase 1 (all CTAs are resident: cooperative launch): quantize this
        // CTA's share of A, then wait for every CTA's share
        const int64_t units = m_tiles * kb;
        if (warp == 0) {
            uint32_t issued = 0;
            if (lane == 0) issued = p1_load(sm, &tmap_x, p, units, kb);
            __syncwarp();
            if (!wait_bands(p, m_tiles, kb, lane)) stop = 1;
            if (lane == 0 && (stop || *static_cast<volatile int*>(&sm.abort_flag))) {
                // let every copy issued into the ring land before the stages are reused or released
                bool landed = true;
                for (uint32_t s = 0; s < kP1Slots && s < issued; ++s) {
                    const uint32_t last = s + kP1Slots * ((issued - 1 - s) / kP1Slots);
                    landed &= wait_plain(smem_u32(&sm.pfull[s]), (last / kP1Slots) & 1, kTeardownLimitNs);
                }
                if (!landed) atomicExch(p.status, kErrTeardown);
                stop = 1;
            }
        }
        if (warp >= 4 && !p1_quantize(sm, p, units, kb, static_cast<int>(threadIdx.x) - 128)) stop = 1;
    }
    tc_fence_before();
    bad = __syncthreads_or(bad);
    if (kFusedA) stop = __syncthreads_or(stop);
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    if (bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(p.status, 0, kErrInvalidArg);
    } else if (stop) {
        // a CTA's share of A never arrived: nothing is computed
    } else if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LOW));
        if (warp == 0 && lane == 0) run_producer<kRowB>(sm, &tmap_a, &tmap_b, p, m_tiles, n_tiles, kb);
        if (warp == 1) run_mma<kRowB>(sm, tmem_base, p, m_tiles, n_tiles, kb, lane);
        if (warp == 2) run_watch<kRowB>(sm, p, m_tiles, n_tiles, kb, lane);
        if constexpr (kRowB != 0)
            if (warp == 3) run_scales(sm, p, m_tiles, n_tiles, kb, lane);
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_HIGH));
        if constexpr (kRowB != 0)
            run_epilogue_rowb(sm, tmem_base, p, &tmap_d, m_tiles, n_tiles, kb, warp, lane);
        else
            run_epilogue(sm, tmem_base, p, &tmap_d, m_tiles, n_tiles, kb, warp, lane);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// -------------------------------------------------------- tensor maps ---
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Tiled map over a K-major uint8 operand [(depth,) rows, K]: box 128 (K) x
// box_rows, 128-byte swizzle, zero fill outside the tensor.
bool encode_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int64_t depth,
                        uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(K) * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const cuuint32_t rank = depth > 0 ? 3 : 2;
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output map over D [M, N] (BF16 or FP32): box of 128 bytes of a row x 32
// rows, 128-byte swizzle (the promotion warps' staging layout).
// Map over a BF16 activation x[M, K] for the fused A quantization: box of
// 64 columns (128 bytes) x 128 rows, 128-byte swizzle.
bool encode_act_map(CUtensorMap* map, const void* base, int64_t M, int64_t K) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_output_map(CUtensorMap* map, void* base, int64_t M, int64_t N, bool bf16) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * esz};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

std::once_flag g_attr_once[64];

}  // namespace

int launch_gemm(const GemmArgs& a, int num_sms, int* status_word, cudaStream_t stream, cudaError_t* cuda_err) {
    *cuda_err = cudaSuccess;
    int dev = 0;
    if ((*cuda_err = cudaGetDevice(&dev)) != cudaSuccess) return kErrCuda;
    if (dev >= 0 && dev < 64) {
        cudaError_t e = cudaSuccess;
        std::call_once(g_attr_once[dev], [&] {
            e = cudaFuncSetAttribute(gemm_blockscaled_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_bytes<0>()));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemm_blockscaled_kernel<1, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<1>()));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gemm_blockscaled_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<0>()));
        });
        if (e != cudaSuccess) {
            *cuda_err = e;
            return kErrCuda;
        }
    }
    CUtensorMap tmap_a, tmap_b, tmap_d, tmap_x;
    std::memset(&tmap_a, 0, sizeof tmap_a);
    std::memset(&tmap_b, 0, sizeof tmap_b);
    std::memset(&tmap_d, 0, sizeof tmap_d);
    std::memset(&tmap_x, 0, sizeof tmap_x);
    if (a.xa && !encode_act_map(&tmap_x, a.xa, a.M, a.K)) return kErrCuda;
    if (!encode_operand_map(&tmap_a, a.a, a.M, a.K, 0, BM)) return kErrCuda;
    if (!encode_operand_map(&tmap_b, a.b, a.N, a.K, a.offsets ? a.G : 0, BN)) return kErrCuda;
    if (!encode_output_map(&tmap_d, a.d, a.M, a.N, a.out_bf16 != 0)) return kErrCuda;
    Params p;
    p.sa = a.sa;
    p.sb = a.sb;
    p.sb_stride_n = a.sb_stride_n;
    p.sb_stride_k = a.sb_stride_k;
    p.sb_group_stride = a.offsets ? (a.N / 128) * (a.K / 128) : 0;
    p.bscale = a.bscale;
    p.d = a.d;
    p.out_bf16 = a.out_bf16;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.offsets = a.offsets;
    p.G = a.G;
    p.m_fastest = a.offsets ? 0 : 1;
    p.status = status_word;
    p.limit_ns = a.wait_limit_ns;
    p.qa = reinterpret_cast<uint2*>(const_cast<uint8_t*>(a.a));
    p.sa_out = const_cast<float*>(a.sa);
    p.band_flags = a.band_flags;
    p.m_tiles = (a.M + BM - 1) / BM;
    const int64_t tiles = p.m_tiles * ((a.N + BN - 1) / BN);
    const int64_t grid = tiles < num_sms ? tiles : num_sms;
    if (grid <= 0) return kOk;
    // the kernel counts a CTA's K chunks (over all its tiles) in 32 bits
    if ((tiles + grid - 1) / grid * (a.K / BK) >= (int64_t(1) << 31)) return kErrInvalidArg;
    if (a.xa) {
        // fused A quantization: the band counters start at zero, and every
        // CTA waits for the others' share of A, so all must be resident at
        // once -- a cooperative launch, which the runtime refuses otherwise
        if ((*cuda_err = cudaMemsetAsync(a.band_flags, 0, static_cast<size_t>(a.M / BM) * sizeof(int32_t),
                                         stream)) != cudaSuccess)
            return kErrCuda;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem_bytes<0>();
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        *cuda_err = cudaLaunchKernelEx(&cfg, gemm_blockscaled_kernel<0, true>, tmap_a, tmap_b, tmap_d, tmap_x, p);
        return *cuda_err == cudaSuccess ? kOk : kErrCuda;
    }
    if (a.bscale == 1)
        gemm_blockscaled_kernel<1, false><<<static_cast<unsigned>(grid), THREADS, smem_bytes<1>(), stream>>>(
            tmap_a, tmap_b, tmap_d, tmap_x, p);
    else
        gemm_blockscaled_kernel<0, false><<<static_cast<unsigned>(grid), THREADS, smem_bytes<0>(), stream>>>(
            tmap_a, tmap_b, tmap_d, tmap_x, p);
    *cuda_err = cudaPeekAtLastError();
    return *cuda_err == cudaSuccess ? kOk : kErrCuda;
}

// ------------------------------------------------- watchdog self-test ---
namespace {
__global__ void watchdog_kernel(uint64_t limit_ns, int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // nobody arrives: the phase never completes and the wait must give up
    if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, limit_ns, kErrTimeout);
    __syncthreads();
}
}  // namespace

cudaError_t launch_watchdog_selftest(uint64_t timeout_ns, int* status_word, cudaStream_t stream) {
    watchdog_kernel<<<1, 32, 0, stream>>>(timeout_ns, status_word);
    return cudaPeekAtLastError();
}

// ------------------------------------------------ tensor-rate probe ---
// The ceiling the block-scaled GEMM is measured against: one CTA per SM
// issues `chunks` x 4 tcgen05.mma.kind::f8f6f4 of 128 x 256 x 32 back to back
// (the GEMM's own instruction shape and operand layout, alternating between
// two 256-column TMEM buffers), with no TMA, no promotion and no output.
// The operands are a fixed pattern of finite E4M3 codes in shared memory.
namespace {
struct __align__(1024) ProbeSmem {
    uint8_t a[A_BYTES];
    uint8_t b[B_BYTES];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int64_t chunks, uint64_t limit_ns, int* status) {
    extern __shared__ uint8_t smem_raw[];
    ProbeSmem& sm =
        *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* words = reinterpret_cast<uint32_t*>(sm.a);
    for (int i = threadIdx.x; i < static_cast<int>((A_BYTES + B_BYTES) / 4); i += blockDim.x)
        words[i] = (0x31u * static_cast<uint32_t>(i) + 0x1234567u) & 0x77777777u;   // no NaN codes
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&sm.done), 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    fence_proxy_async_shared();
    if (warp == 0) tmem_alloc(smem_u32(&sm.tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t adesc = smem_desc_sw128(smem_u32(sm.a));
            const uint64_t bdesc = smem_desc_sw128(smem_u32(sm.b));
            for (int64_t c = 0; c < chunks; ++c) {
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(c & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < BK / MMA_K; ++kk) {
                    const uint64_t koff = static_cast<uint64_t>((kk * MMA_K) >> 4);
                    mma_f8f6f4(d_tmem, adesc + koff, bdesc + koff, kIdesc, kk > 0 ? 1u : 0u);
                }
            }
            mma_commit(smem_u32(&sm.done));
            if (!mbar_wait_bounded(smem_u32(&sm.done), 0, &sm.abort_flag, status, limit_ns, kErrTimeout)) {
                // the MMAs must finish before TMEM is released
                if (!wait_plain(smem_u32(&sm.done), 0, 10 * kTeardownLimitNs)) atomicExch(status, kErrTeardown);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base, TMEM_COLS);
}
std::once_flag g_probe_attr_once[64];
}  // namespace

cudaError_t launch_mma_rate_probe(int64_t chunks, int num_sms, uint64_t limit_ns, int* status_word,
                                  cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // more than half of an SM's shared memory: one probe CTA per SM
    const int smem = static_cast<int>(sizeof(ProbeSmem) + 1024) > 120 * 1024 ? static_cast<int>(sizeof(ProbeSmem) + 1024)
                                                                                : 120 * 1024;
    if (dev >= 0 && dev < 64) {
        std::call_once(g_probe_attr_once[dev], [&] {
            e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        });
        if (e != cudaSuccess) return e;
    }
    mma_rate_kernel<<<num_sms, 128, smem, stream>>>(chunks, limit_ns, status_word);
    return cudaPeekAtLastError();
}

}  // namespace fp8fg
