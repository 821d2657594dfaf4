// Tensor-core GEMMs on tcgen05 (sm_103a): the scaled FP8 GEMM and the exact
// INT8 GEMM with its per-row x per-row dequantization epilogue.
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: streams 128x128-byte A tiles and BNx128-byte B
//               tiles (128-byte swizzle) into a ring of shared-memory stages.
//   warp 1      owns the TMEM allocation; one elected thread issues
//               tcgen05.mma (M=128, N=BN, K=32 bytes per instruction) into one
//               of two TMEM accumulators and releases each stage with
//               tcgen05.commit.
//   warps 2..   epilogue: tcgen05.ld of the accumulator, scaling, stores.  Two
//               accumulators let the epilogue of one tile overlap the MMAs of
//               the next.
// Tiles are visited in groups of GROUP_M tile-rows so that consecutive CTAs
// share B column blocks in L2 (grouped rasterisation, as the AstrAI commit
// notes do for the NT forward).
//
// FP8 (AstrAI ops/fp8.py, custom::fp8_gemm): acc = sum_k a8*b8 in FP32 inside
// the tensor core (kind::f8f6f4, E4M3 or E5M2), C = bf16(fl32(acc*sa)*sb).
// NT, NN and TN are served by the same kernel: an operand stored with M (or
// N) contiguous is loaded as [K rows x 128 bytes] boxes and described to the
// MMA as MN-major, so no transposed copy is ever made.
//
// INT8 (scmp_kernels sc_matmul per_row / per_head, C = a @ b.T in float32):
// sm_103a has no kind::i8, so the codes are staged as fp16 (exact for
// |q| <= 127) and multiplied with kind::f16 into an FP32 accumulator.  Every
// product is an integer of magnitude <= 127^2 and every partial sum of a
// 1024-long K chunk is an integer below 127^2 * 1024 < 2^24, so the FP32
// accumulation of a chunk is exact.  The epilogue converts each chunk to int32
// and sums the chunks in registers, which keeps the whole K sum exact.
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "sq_device.cuh"
#include "sq_host.h"
#include "sq_launch.h"

namespace sq {

constexpr int kBM = 128;
constexpr int kBKBytes = 128;   // bytes of K per stage row (one 128-B swizzle row)
constexpr int kGroupM = 16;      // FP8: tile rows per raster group
constexpr int kGroupMI8 = 8;     // INT8: its 16-bit operand stripes are twice as large
constexpr int kI8ChunkK = 1024; // K elements per exact FP32 chunk
constexpr int kStgChunk = 1024; // codes per warp chunk of the INT8 staging pipeline
constexpr int kStgMaxParts = 256; // staging CTAs per operand (each writes one bound slot)

struct GemmParams {
    int M, N, K;
    int batch;
    int mt, nt;            // tile counts along M and N
    int nkb;               // k-blocks per tile
    int kb_per_chunk;      // k-blocks per accumulator chunk
    int nchunks;
    const float* sa;       // FP8: scalar step of A; INT8: row scales [batch*M]
    const float* sb;       // FP8: scalar step of B; INT8: row scales [batch*N]
    void* C;               // FP8: bf16 [M,N]; INT8: f32, batch stride strideC
    int32_t* acc_out;      // INT8 only (nullable)
    int group_m;           // tile rows per raster group
    int tma_store;         // FP8 bf16 output: stage 32x32 boxes in shared memory, store with TMA
    // INT8: the bound regions that the staging wrote in the workspace
    // (sq_bound.h layout: a header word, then one slot per staging CTA), and
    // how many staged chunks of kStgChunk codes one row can overlap
    const unsigned* bound_a;
    const unsigned* bound_b;
    int row_chunks_a, row_chunks_b;
    int64_t strideC;
    uint32_t idesc;
    int vec_store;
    unsigned* err_word;
    const float* out_scale; // FP8 with E4M3 output: the output step (divided out)
    int out_e4m3;           // FP8: 1 = C is E4M3 codes [M,N], 0 = bf16
    int ga, gb;             // INT8: rows per scale group of A and B (1 = per row)
    int Mg, Ng;             // INT8: scale groups per batch, ceil(M/ga), ceil(N/gb)
    int sb_vec;             // INT8: sB may be read 4 floats at a time
    const float* bias;      // FP8: float32 bias per output column, added after scaling (nullable)
    // Diagnostics (nullable): per CTA, SM cycles and %globaltimer at entry
    // and at exit, [cycles0, cycles1, ns0, ns1], for CTAs below clk_cap
    unsigned long long* clk;
    int clk_cap;
    // Grouped FP8 launches: this problem's operand layouts (1 = stored with M,
    // or N, contiguous), which the other launches take from the template
    int a_mn, b_mn;
};

// PAIR = false: one CTA per SM computes 128 x BN tiles (cta_group::1).
// PAIR = true:  a cluster of two CTAs on the two SMs of a TPC computes
//               256 x BN tiles with cta_group::2 MMAs issued by the leader
//               (rank 0): each CTA holds 128 rows of A and BN/2 rows of B, so
//               each SM reads half of the B tile from its shared memory.
template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI>
struct GemmCfg {
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;           // B rows this CTA stages
    static constexpr int A_BYTES = kBM * kBKBytes;              // 16 KB
    static constexpr int B_BYTES = B_ROWS * kBKBytes;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    // INT8 pair/128-wide tiles take a 7th stage (no output staging buffer there)
    static constexpr int STAGES = (STAGE >= 48 * 1024) ? 4 : (I8 ? 7 : 6);
    static constexpr int TILE_M = PAIR ? 2 * kBM : kBM;
    // Epilogue warps, each owning 32 rows x EPI_COLS columns of the tile.
    // INT8 keeps its running int32 sums in registers, so it takes 8.  FP8
    // takes 8 on 128-wide tiles, where one tile per CTA leaves the epilogue
    // exposed (5-7% faster on one-wave shapes), and on 256-wide tiles of
    // launches that run a single round of tiles (WIDE_EPI); 4 on 256-wide
    // tiles of longer launches, whose epilogue overlaps the next tile's MMAs
    // (8 measured about 1% slower there).  32-wide INT8 tiles take 4, one
    // 32-column slice each.
    static constexpr int EPI_WARPS = BN == 32 ? 4 : ((I8 || BN == 128 || WIDE_EPI) ? 8 : 4);
    static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    // FP8: two 32 x 32 bf16 output boxes (2 KB each) per epilogue warp
    static constexpr int EPI_STAGE = I8 ? 0 : EPI_WARPS * 2 * 2048;
    static constexpr int SMEM = STAGES * STAGE + EPI_STAGE + BAR_BYTES + 1024;
    // bytes the start address moves per MMA instruction along K
    static constexpr int KSTEP_K = 32;                      // K-major: 32 B inside the row
    static constexpr int KSTEP_MN = (I8 ? 16 : 32) * 128;   // MN-major: that many K rows
    static constexpr int MN_LBO = kBKBytes * 128;           // 16 KB between 128-B column blocks
    static_assert(2 * STAGES * 8 + 5 * 8 + 24 <= BAR_BYTES, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
    // the TMEM allocation is made before the grid-dependency wait, which
    // relies on no two GEMM CTAs (of any shape) sharing an SM
    static_assert(2 * (SMEM + 1024) > 233472, "one GEMM CTA per SM");
    static_assert(!B_MN || B_ROWS % 128 == 0, "MN-major B is staged in 128-column blocks");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& b, int& mb, int& nb) {
    const int per = p.mt * p.nt;
    b = t / per;
    const int r = t - b * per;
    const int gsz = p.group_m * p.nt;
    const int g = r / gsz;
    const int first = g * p.group_m;
    const int gm = min(p.mt - first, p.group_m);
    const int rr = r - g * gsz;
    mb = first + rr % gm;
    nb = rr / gm;
}

// Two floats to two bf16 (RN) in one word, lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Per-CTA state that the warp roles of gemm_tc_kernel share: pointers into
// shared memory, the TMEM base, this CTA's identity and its tile range.
struct GemmCta {
    uint8_t* smem;              // operand stages (1024-aligned)
    uint8_t* epi_stage;         // FP8: output staging boxes
    uint64_t* full;             // [STAGES] stage landed
    uint64_t* empty;            // [STAGES] stage consumed by the MMAs
    uint64_t* tfull;            // [2] accumulator complete
    uint64_t* tempty;           // [2] accumulator read by every epilogue warp
    uint64_t* drain;            // MMAs issued before an abort have finished
    volatile int* abort_flag;
    uint32_t tmem_base;
    uint32_t rank;              // 0 = leader of the pair
    bool leader;
    int cta_unit, num_units;    // this CTA's (or pair's) index and their count
    int total;                  // tiles in the launch
    int total0;                 // grouped launches: tiles of the first problem (else total)
};

// The unit a CTA (or pair) takes in its r-th round of the tile loop.  Grouped
// launches alternate the rounds' direction, so that the CTAs whose first unit
// was a long tile of the first problem take the later rounds' units last.
template <bool GRP>
__device__ __forceinline__ int unit_of(int r, const GemmCta& c) {
    return r * c.num_units + ((GRP && (r & 1)) ? c.num_units - 1 - c.cta_unit : c.cta_unit);
}

// The unit of round r, given t, the unit of round r - 1.
template <bool GRP>
__device__ __forceinline__ int next_unit(int t, int r, const GemmCta& c) {
    return GRP ? unit_of<true>(r, c) : t + c.num_units;
}

// Warp 0: one elected thread streams the A and B boxes of every k-block of
// this CTA's tiles into the ring of stages.
template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI, bool GRP>
__device__ __forceinline__ void gemm_producer(const CUtensorMap* tmAs, const CUtensorMap* tmBs,
                                              const GemmParams* P, const GemmCta& c) {
    using Cfg = GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    uint8_t* smem = c.smem;
    uint64_t* full = c.full;
    uint64_t* empty = c.empty;
    volatile int* abort_flag = c.abort_flag;
    const uint32_t rank = c.rank;
    const bool leader = c.leader;
    const int total = c.total;
    if (elect_one_sync()) {
        int stage = 0;
        uint32_t phase = 0;
        int issued_phase[Cfg::STAGES];
        for (int s = 0; s < Cfg::STAGES; ++s) issued_phase[s] = -1;
        bool ok = true;
        bool first_round = true;   // the ring's stages are all free until it wraps
        bool waited = false;
        for (int r = 0, t = c.cta_unit; t < total && ok; t = next_unit<GRP>(t, ++r, c)) {
            const int pi = (GRP && t >= c.total0) ? 1 : 0;
            const GemmParams& p = P[pi];
            const CUtensorMap& tmA = tmAs[pi];
            const CUtensorMap& tmB = tmBs[pi];
            const bool a_mn = GRP ? p.a_mn != 0 : A_MN;
            const bool b_mn = GRP ? p.b_mn != 0 : B_MN;
            int b, mb, nb;
            tile_coords(t - (pi ? c.total0 : 0), p, b, mb, nb);
            const int m0 = mb * Cfg::TILE_M + static_cast<int>(rank) * kBM;
            const int n0 = nb * BN + static_cast<int>(rank) * Cfg::B_ROWS;
            for (int kb = 0; kb < p.nkb; ++kb) {
                if (!first_round && !mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.err_word)) {
                    ok = false;
                    break;
                }
                uint8_t* sA = smem + stage * Cfg::STAGE;
                uint8_t* sB = sA + Cfg::A_BYTES;
                if (PAIR) {
                    // both CTAs' bytes complete on the leader's barrier
                    const uint32_t fb = cluster_addr(&full[stage], 0);
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * Cfg::STAGE);
                    if (!waited) {
                        pdl_wait();   // the operands are the previous kernels' output
                        waited = true;
                    }
                    if (I8) {
                        const int kx = kb * (kBKBytes / 2);
                        tma_load_3d_pair(sA, &tmA, fb, kx, m0, b);
                        tma_load_3d_pair(sB, &tmB, fb, kx, n0, b);
                    } else {
                        const int kx = kb * kBKBytes;
                        if (a_mn) tma_load_2d_pair(sA, &tmA, fb, m0, kx);
                        else tma_load_2d_pair(sA, &tmA, fb, kx, m0);
                        if (b_mn) {
#pragma unroll
                            for (int j = 0; j < Cfg::B_ROWS / 128; ++j)
                                tma_load_2d_pair(sB + j * Cfg::MN_LBO, &tmB, fb, n0 + j * 128, kx);
                        } else {
                            tma_load_2d_pair(sB, &tmB, fb, kx, n0);
                        }
                    }
                } else {
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE);
                    if (!waited) {
                        pdl_wait();   // the operands are the previous kernels' output
                        waited = true;
                    }
                    if (I8) {
                        const int kx = kb * (kBKBytes / 2);
                        tma_load_3d(sA, &tmA, &full[stage], kx, m0, b);
                        tma_load_3d(sB, &tmB, &full[stage], kx, n0, b);
                    } else {
                        const int kx = kb * kBKBytes;
                        if (a_mn) tma_load_2d(sA, &tmA, &full[stage], m0, kx);
                        else tma_load_2d(sA, &tmA, &full[stage], kx, m0);
                        if (b_mn) {
#pragma unroll
                            for (int j = 0; j < Cfg::B_ROWS / 128; ++j)
                                tma_load_2d(sB + j * Cfg::MN_LBO, &tmB, &full[stage], n0 + j * 128, kx);
                        } else {
                            tma_load_2d(sB, &tmB, &full[stage], kx, n0);
                        }
                    }
                }
                issued_phase[stage] = static_cast<int>(phase);
                if (++stage == Cfg::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                    first_round = false;
                }
            }
        }
        if (!ok && leader) {
            // let every copy signalled on this CTA's barriers land before it exits
            for (int s = 0; s < Cfg::STAGES; ++s)
                if (issued_phase[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]));
        }
    }
}

// Warp 1: on the leader, one elected thread issues the MMAs of each k-block
// into one of the two TMEM accumulators (kbpc k-blocks per accumulator
// chunk, nch chunks per tile) and commits stages and accumulators.
template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI, bool GRP>
__device__ __forceinline__ void gemm_mma(const GemmParams* P, const GemmCta& c, int kbpc, int nch) {
    using Cfg = GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    uint8_t* smem = c.smem;
    uint64_t* full = c.full;
    uint64_t* empty = c.empty;
    uint64_t* tfull = c.tfull;
    uint64_t* tempty = c.tempty;
    uint64_t* drain = c.drain;
    volatile int* abort_flag = c.abort_flag;
    const uint32_t tmem_base = c.tmem_base;
    const bool leader = c.leader;
    const int total = c.total;
    if (leader && elect_one_sync()) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t it = 0;
        bool ok = true;
        bool issued = false;
        for (int r = 0, t = c.cta_unit; t < total && ok; t = next_unit<GRP>(t, ++r, c)) {
            const GemmParams& p = P[(GRP && t >= c.total0) ? 1 : 0];
            const bool a_mn = GRP ? p.a_mn != 0 : A_MN;
            const bool b_mn = GRP ? p.b_mn != 0 : B_MN;
            // FP8 takes the whole K in one accumulator chunk
            const int tkbpc = I8 ? kbpc : p.nkb;
            const int tnch = I8 ? nch : 1;
            for (int ch = 0; ch < tnch && ok; ++ch) {
                const uint32_t ab = it & 1u;
                const uint32_t aph = (it >> 1) & 1u;
                if (!mbar_wait(&tempty[ab], aph ^ 1u, abort_flag, p.err_word)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + ab * BN;
                const int kb0 = ch * tkbpc;
                const int kb1 = min(p.nkb, kb0 + tkbpc);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.err_word)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(smem + stage * Cfg::STAGE);
                    const uint32_t b_addr = a_addr + Cfg::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBKBytes / 32; ++kk) {
                        const uint64_t ad =
                            a_mn ? sdesc_sw128(a_addr + kk * Cfg::KSTEP_MN, Cfg::MN_LBO, 1024)
                                 : sdesc_sw128(a_addr + kk * Cfg::KSTEP_K, 16, 1024);
                        const uint64_t bd =
                            b_mn ? sdesc_sw128(b_addr + kk * Cfg::KSTEP_MN, Cfg::MN_LBO, 1024)
                                 : sdesc_sw128(b_addr + kk * Cfg::KSTEP_K, 16, 1024);
                        const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
                        if (PAIR) {
                            if (I8) mma_pair_f16(d_tmem, ad, bd, p.idesc, acc);
                            else mma_pair_f8f6f4(d_tmem, ad, bd, p.idesc, acc);
                        } else {
                            if (I8) mma_f16(d_tmem, ad, bd, p.idesc, acc);
                            else mma_f8f6f4(d_tmem, ad, bd, p.idesc, acc);
                        }
                    }
                    issued = true;
                    if (PAIR) mma_commit_pair(&empty[stage], 3);   // frees the stage in both CTAs
                    else mma_commit(&empty[stage]);
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (PAIR) mma_commit_pair(&tfull[ab], 3);          // both epilogues may read
                else mma_commit(&tfull[ab]);
                ++it;
            }
        }
        if (!ok && issued) {
            // make every MMA already issued finish before TMEM is released
            if (PAIR) mma_commit_pair(drain, 1);
            else mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    }
}

// Warps 2..: read each finished accumulator out of TMEM, scale it and store
// the tile (INT8: int32 sums of nch chunks, fp32 dequantized output; FP8:
// bf16 or E4M3 output).
// On CTA pairs the FP8 epilogue arrives on the cluster barrier (the one that
// precedes the TMEM release) as soon as it has read its last accumulator, so
// that the barrier completes while it converts and stores; it returns whether
// it has arrived.
template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI, bool GRP>
__device__ __forceinline__ bool gemm_epilogue(const CUtensorMap* tmCs, const GemmParams* P,
                                              const GemmCta& c, int nch) {
    using Cfg = GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* smem = c.smem;
    uint8_t* epi_stage = c.epi_stage;
    uint64_t* tfull = c.tfull;
    uint64_t* tempty = c.tempty;
    volatile int* abort_flag = c.abort_flag;
    const uint32_t tmem_base = c.tmem_base;
    const uint32_t rank = c.rank;
    const bool leader = c.leader;
    const int total = c.total;
    const int ew = warp - 2;
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int colgrp = ew >> 2;            // which EPI_COLS-wide column group
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // where this warp reports that it has read an accumulator: the leader's barrier
    const uint32_t tempty_leader[2] = {PAIR ? cluster_addr(&tempty[0], 0) : 0u,
                                       PAIR ? cluster_addr(&tempty[1], 0) : 0u};
    // FP8: each problem's two steps (grouped launches: bf16 outputs only)
    float fsa2[2] = {0.0f, 0.0f}, fsb2[2] = {0.0f, 0.0f}, fos = 1.0f, foy = 1.0f;
    bool ofast = true;
    if (!I8) {
        fsa2[0] = *P[0].sa;
        fsb2[0] = *P[0].sb;
        if (GRP) {
            fsa2[1] = *P[1].sa;
            fsb2[1] = *P[1].sb;
        }
        if (P[0].out_e4m3) {
            fos = *P[0].out_scale;
            foy = __frcp_rn(fos);
            ofast = fos >= 0x1p-40f && fos <= 0x1p40f;
        }
    }
    uint32_t it = 0;
    uint32_t sc = 0;                       // output boxes this warp has stored
    bool ok = true;
    bool arrived = false;
    auto release = [&](uint32_t ab) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (PAIR && !leader) mbar_arrive_cluster(tempty_leader[ab]);
            else mbar_arrive(&tempty[ab]);
        }
    };
    for (int r = 0, t = c.cta_unit; t < total && ok; t = next_unit<GRP>(t, ++r, c)) {
        const int pi = (GRP && t >= c.total0) ? 1 : 0;
        const GemmParams& p = P[pi];
        const CUtensorMap& tmC = tmCs[pi];
        const float fsa = fsa2[pi], fsb = fsb2[pi];
        const bool last = next_unit<GRP>(t, r + 1, c) >= total;   // this CTA's last tile
        int b, mb, nb;
        tile_coords(t - (pi ? c.total0 : 0), p, b, mb, nb);
        const int m0 = mb * Cfg::TILE_M + static_cast<int>(rank) * kBM;
        const int n0 = nb * BN;
        const int row = m0 + quarter * 32 + lane;
        if (I8) {
            constexpr int NC = Cfg::EPI_COLS / 32;
            // A CTA's last tile: every MMA has completed and no TMA load is
            // pending once its last accumulator is read, so the operand
            // stages are free.  Each warp stages its 32 rows there and then
            // writes whole row runs (one 512-byte run, or two 256-byte ones,
            // per instruction) instead of a 16-byte piece in each of 32
            // rows.  On one-wave problems this store is the exposed tail of
            // the kernel, so its scales are loaded before the accumulator
            // is waited for.
            constexpr int PITCH = Cfg::EPI_COLS + 4;   // int32 words per staged row
            constexpr int F4_ROW = Cfg::EPI_COLS / 4;   // 16-byte pieces per row
            constexpr int ROWS_STEP = 32 / F4_ROW;      // rows one warp-wide store covers
            static_assert(Cfg::EPI_WARPS * 32 * PITCH * 4 <= Cfg::STAGES * Cfg::STAGE,
                          "staged output fits in the operand stages");
            const bool staged = p.vec_store && last;
            const int scol = n0 + colgrp * Cfg::EPI_COLS + 4 * (lane % F4_ROW);
            const bool scol_ok = scol < p.N;   // N % 4 == 0: all four columns are in range
            float st_sa = 0.0f;
            float4 st_sb = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (staged) {
                if (row < p.M) st_sa = p.sa[static_cast<int64_t>(b) * p.Mg + row / p.ga];
                if (p.C && scol_ok) {
                    const float* sBb = p.sb + static_cast<int64_t>(b) * p.Ng;
                    if (p.sb_vec) {
                        st_sb = *reinterpret_cast<const float4*>(sBb + scol);
                    } else {
                        st_sb.x = sBb[scol / p.gb];
                        st_sb.y = sBb[(scol + 1) / p.gb];
                        st_sb.z = sBb[(scol + 2) / p.gb];
                        st_sb.w = sBb[(scol + 3) / p.gb];
                    }
                }
            }
            // One chunk (the whole K summed exactly in fp32): the sums keep the
            // accumulator's bits, each an exact integer, and become int32 only
            // where acc_out asks for one; C takes the float itself (+0 for a
            // zero sum, as float(0) is).  The float-to-int conversions, a slow
            // pipe, then stay off a one-wave kernel's exposed tail.  Several
            // chunks: each is converted and added in int32.
            const bool raw = nch == 1;
            auto as_f = [&](int32_t v) {
                return raw ? __fadd_rn(__int_as_float(v), 0.0f) : __int2float_rn(v);
            };
            auto as_i = [&](int32_t v) { return raw ? __float2int_rn(__int_as_float(v)) : v; };
            int32_t sums[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) sums[c][i] = 0;
            for (int ch = 0; ch < nch; ++ch) {
                const uint32_t ab = it & 1u;
                const uint32_t aph = (it >> 1) & 1u;
                if (!mbar_wait(&tfull[ab], aph, abort_flag, p.err_word)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem_base + lane_off + ab * BN + colgrp * Cfg::EPI_COLS;
                if (raw) {
                    // every column of this warp in flight behind one wait
#pragma unroll
                    for (int c = 0; c < NC; ++c)
                        tmem_ld32(tb + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sums[c][0]));
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t r[16];
                            tmem_ld16(tb + c * 32 + h * 16, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                sums[c][h * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                        }
                    }
                }
                release(ab);
                ++it;
            }
            if (!ok) break;
            if (staged) {
                int32_t* stg = reinterpret_cast<int32_t*>(smem) + ew * 32 * PITCH;
                fence_proxy_async_smem();
#pragma unroll
                for (int c = 0; c < NC; ++c)
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        *reinterpret_cast<int4*>(stg + lane * PITCH + c * 32 + 4 * v) =
                            make_int4(sums[c][4 * v], sums[c][4 * v + 1], sums[c][4 * v + 2],
                                      sums[c][4 * v + 3]);
                __syncwarp();
                const int j = lane % F4_ROW;
                float* Cf = static_cast<float*>(p.C);
                const float4 s4 = st_sb;
#pragma unroll 4
                for (int r0 = 0; r0 < 32; r0 += ROWS_STEP) {
                    const int r = r0 + lane / F4_ROW;
                    const float sr = __shfl_sync(0xffffffffu, st_sa, r);
                    const int grow = m0 + quarter * 32 + r;
                    if (grow < p.M && scol_ok) {
                        const int4 a = *reinterpret_cast<const int4*>(stg + r * PITCH + 4 * j);
                        const int64_t o = static_cast<int64_t>(b) * p.strideC +
                                          static_cast<int64_t>(grow) * p.N + scol;
                        if (p.acc_out)
                            st_v4(p.acc_out + o, make_uint4(as_i(a.x), as_i(a.y), as_i(a.z), as_i(a.w)));
                        if (Cf)
                            st_v4(Cf + o, make_uint4(
                                __float_as_uint(__fmul_rn(__fmul_rn(as_f(a.x), sr), s4.x)),
                                __float_as_uint(__fmul_rn(__fmul_rn(as_f(a.y), sr), s4.y)),
                                __float_as_uint(__fmul_rn(__fmul_rn(as_f(a.z), sr), s4.z)),
                                __float_as_uint(__fmul_rn(__fmul_rn(as_f(a.w), sr), s4.w))));
                    }
                }
            } else if (row < p.M) {
                const float sArow = p.sa[static_cast<int64_t>(b) * p.Mg + row / p.ga];
                const float* sBb = p.sb + static_cast<int64_t>(b) * p.Ng;
                const int64_t obase = static_cast<int64_t>(b) * p.strideC + static_cast<int64_t>(row) * p.N;
                float* Cf = static_cast<float*>(p.C);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int col0 = n0 + colgrp * Cfg::EPI_COLS + c * 32;
                    if (p.vec_store && col0 + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            float4 s4;
                            if (p.sb_vec) {
                                s4 = *reinterpret_cast<const float4*>(sBb + col0 + 4 * v);
                            } else {
                                s4.x = sBb[(col0 + 4 * v) / p.gb];
                                s4.y = sBb[(col0 + 4 * v + 1) / p.gb];
                                s4.z = sBb[(col0 + 4 * v + 2) / p.gb];
                                s4.w = sBb[(col0 + 4 * v + 3) / p.gb];
                            }
                            const int32_t a0 = sums[c][4 * v], a1 = sums[c][4 * v + 1];
                            const int32_t a2 = sums[c][4 * v + 2], a3 = sums[c][4 * v + 3];
                            if (p.acc_out)
                                st_v4(p.acc_out + obase + col0 + 4 * v,
                                      make_uint4(as_i(a0), as_i(a1), as_i(a2), as_i(a3)));
                            if (Cf) {
                                float4 o;
                                o.x = __fmul_rn(__fmul_rn(as_f(a0), sArow), s4.x);
                                o.y = __fmul_rn(__fmul_rn(as_f(a1), sArow), s4.y);
                                o.z = __fmul_rn(__fmul_rn(as_f(a2), sArow), s4.z);
                                o.w = __fmul_rn(__fmul_rn(as_f(a3), sArow), s4.w);
                                st_v4(Cf + obase + col0 + 4 * v,
                                      make_uint4(__float_as_uint(o.x), __float_as_uint(o.y),
                                                 __float_as_uint(o.z), __float_as_uint(o.w)));
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int col = col0 + i;
                            if (col < p.N) {
                                if (p.acc_out) p.acc_out[obase + col] = as_i(sums[c][i]);
                                if (Cf)
                                    Cf[obase + col] = __fmul_rn(__fmul_rn(as_f(sums[c][i]), sArow),
                                                                sBb[col / p.gb]);
                            }
                        }
                    }
                }
            }
        } else {
            const uint32_t ab = it & 1u;
            const uint32_t aph = (it >> 1) & 1u;
            if (!mbar_wait(&tfull[ab], aph, abort_flag, p.err_word)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem_base + lane_off + ab * BN + colgrp * Cfg::EPI_COLS;
            uint16_t* Cb = static_cast<uint16_t*>(p.C);
            const int64_t obase = static_cast<int64_t>(row) * p.N;
            // A CTA's last tile: its MMAs have completed and no TMA load is
            // pending, so the operand stages are free.  Each warp gives every
            // one of its output boxes its own 2 KB there, and no box waits
            // for an earlier box's store to be read (on one-wave problems this
            // epilogue is the kernel's exposed tail).
            const bool last_staged = p.tma_store && !p.out_e4m3 && last;
            static_assert(Cfg::EPI_WARPS * (Cfg::EPI_COLS / 32) * 2048 <= Cfg::STAGES * Cfg::STAGE,
                          "a last tile's output boxes fit in the operand stages");
            int box = 0;
            if (last_staged) fence_proxy_async_smem();
            // one 32-column piece of this warp's 32 rows: scale, round, store
            auto emit = [&](uint32_t (&r)[32], const int col0) {
                if (p.bias && row < p.M) {
                    // bias fused into the epilogue: fl32(fl32(acc*sa)*sb) + bias[col]
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = col0 + i;
                        const float bj = col < p.N ? p.bias[col] : 0.0f;
                        r[i] = __float_as_uint(__fadd_rn(
                            __fmul_rn(__fmul_rn(__uint_as_float(r[i]), fsa), fsb), bj));
                    }
                }
                const float esa = p.bias ? 1.0f : fsa;   // scaling already applied above
                const float esb = p.bias ? 1.0f : fsb;
                if (row < p.M && p.out_e4m3) {
                    // E4M3 output: code = e4m3(fl32(fl32(acc*sa)*sb) / out_scale)
                    uint8_t* C8 = static_cast<uint8_t*>(p.C);
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float w = __fmul_rn(__fmul_rn(__uint_as_float(r[4 * i + e]), esa), esb);
                            v[e] = ofast ? fp8_quotient(w, fos, foy) : __fdiv_rn(w, fos);
                        }
                        pk[i] = fp8x2<0>(v[0], v[1]) | (fp8x2<0>(v[2], v[3]) << 16);
                    }
                    if (p.vec_store && col0 + 32 <= p.N) {
                        st_v4(C8 + obase + col0, make_uint4(pk[0], pk[1], pk[2], pk[3]));
                        st_v4(C8 + obase + col0 + 16, make_uint4(pk[4], pk[5], pk[6], pk[7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + i < p.N)
                                C8[obase + col0 + i] = static_cast<uint8_t>(pk[i >> 2] >> (8 * (i & 3)));
                    }
                } else if (!p.out_e4m3 && p.tma_store) {
                    // The warp's 32 rows x 32 columns go out as one TMA box: each
                    // lane writes its 64-byte row into a 64-byte-swizzled staging
                    // buffer (16-byte piece j of row r sits at piece j ^ ((r >> 1) & 3),
                    // which keeps the writes conflict-free); rows or columns past
                    // the matrix are clipped by the store.
                    uint8_t* buf;
                    if (last_staged) {
                        buf = smem + (ew * (Cfg::EPI_COLS / 32) + box++) * 2048;
                    } else {
                        buf = epi_stage + (ew * 2 + (sc & 1u)) * 2048;
                        if (lane == 0 && sc >= 2) bulk_wait_read<1>();   // the box two back is read
                        __syncwarp();
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = bf16x2_bits(__fmul_rn(__fmul_rn(__uint_as_float(r[2 * i]), esa), esb),
                                            __fmul_rn(__fmul_rn(__uint_as_float(r[2 * i + 1]), esa), esb));
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    ++sc;
                    // a last tile's boxes are stored together after the loop,
                    // behind one proxy fence
                    if (last_staged) return;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, col0, m0 + quarter * 32);
                        bulk_commit();
                    }
                } else if (row < p.M) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float lo = __fmul_rn(__fmul_rn(__uint_as_float(r[2 * i]), esa), esb);
                        const float hi = __fmul_rn(__fmul_rn(__uint_as_float(r[2 * i + 1]), esa), esb);
                        pk[i] = bf16x2_bits(lo, hi);
                    }
                    if (p.vec_store && col0 + 32 <= p.N) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            st_v4(Cb + obase + col0 + 8 * v,
                                  make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + i < p.N)
                                Cb[obase + col0 + i] =
                                    static_cast<uint16_t>((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xFFFFu));
                    }
                }
            };
#pragma unroll 1
            for (int c = 0; c < Cfg::EPI_COLS / 32; c += 2) {
                // two TMEM loads in flight behind one wait
                uint32_t r0[32], r1[32];
                tmem_ld32(tb + c * 32, r0);
                tmem_ld32(tb + (c + 1) * 32, r1);
                tmem_ld_wait();
                if (PAIR && last && c + 2 >= Cfg::EPI_COLS / 32) {
                    // this warp's last read of TMEM, and no accumulator is
                    // released after the last tile: nothing of this warp
                    // touches the peer CTA or TMEM any more
                    tc_fence_before();
                    cluster_arrive();
                    arrived = true;
                }
                const int col0 = n0 + colgrp * Cfg::EPI_COLS + c * 32;
                emit(r0, col0);
                emit(r1, col0 + 32);
            }
            if (last_staged) {
                // the shared-memory writes of every box, then their stores
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    for (int b = 0; b < box; ++b)
                        tma_store_2d(&tmC, smem + (ew * (Cfg::EPI_COLS / 32) + b) * 2048,
                                     n0 + colgrp * Cfg::EPI_COLS + b * 32, m0 + quarter * 32);
                    bulk_commit();
                }
            }
            // the MMA warp waits for a released accumulator only before a
            // next tile
            if (!last) release(ab);
            ++it;
        }
    }
    // the staged output boxes must be written (and their buffers read) before exit
    if (!I8 && lane == 0 && sc > 0) bulk_wait_all();
    return arrived;
}

// The kernel body: P[0] (and on grouped launches P[1]) with their maps;
// units [0, total0) are tiles of the first problem, [total0, total) of the
// second.
template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI, bool GRP>
__device__ __forceinline__ void gemm_body(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                          const CUtensorMap* tmC, const GemmParams* P, int total0,
                                          int total) {
    using Cfg = GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    const GemmParams& p = P[0];
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* epi_stage = smem + Cfg::STAGES * Cfg::STAGE;     // 1024-aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(epi_stage + Cfg::EPI_STAGE);
    uint64_t* empty = full + Cfg::STAGES;
    uint64_t* tfull = empty + Cfg::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned* bound_max = reinterpret_cast<unsigned*>(tmem_slot + 2);   // INT8: [A, B, mult A, mult B]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned long long clk0 = 0, ns0 = 0;
    if (p.clk && threadIdx.x == 0) {
        clk0 = clock64();
        ns0 = global_ns_ordered();
    }
    const uint32_t rank = PAIR ? cluster_rank() : 0u;   // 0 = leader of the pair
    const bool leader = rank == 0;
    const int cta_unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int num_units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], (PAIR ? 2 : 1) * Cfg::EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int i = 0; i < (GRP ? 2 : 1); ++i) {
            tma_prefetch_desc(&tmA[i]);
            tma_prefetch_desc(&tmB[i]);
            if (!I8 && P[i].tma_store) tma_prefetch_desc(&tmC[i]);
        }
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    // Nothing above or in the shared set-up below reads or writes global
    // memory, so it all overlaps the previous kernel's tail.  (No two GEMM
    // CTAs fit on one SM, so the allocation never waits for an earlier GEMM's
    // TMEM.)  Each role waits for the previous kernel right before its own
    // first global access: the producer once its first stage is armed, the
    // other warps below, thread 0 again before its clock record.
    pdl_allow_next();
    tc_fence_before();
    __syncthreads();
    if (PAIR) {
        __syncwarp();
        cluster_sync_all();   // the peer's barriers exist before anyone signals them
    }
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // INT8 exactness.  Every partial sum the tensor core forms for C[i,j] is an
    // integer of magnitude at most sum_k |a_ik b_jk| <= |a_i|_2 |b_j|_2
    // (Cauchy-Schwarz).  The staging bounds |a_i|_2^2 either by the largest
    // row norm itself or by row_chunks_a * (the largest sum of squares over a
    // staged chunk).  When the product of the two bounds is below 2^48, every
    // partial sum stays below 2^24 and is exact in fp32 in any order, so the
    // whole K is accumulated in one chunk; otherwise the accumulator is
    // drained into int32 every kI8ChunkK (127^2 * 1024 < 2^24).
    //
    // Only the MMA issuer and the epilogue need the decision: warps 2 and 3
    // read the bounds while the producer already streams the first stages,
    // and a named barrier among warps 1.. hands the result over.
    if (warp != 0) pdl_wait();
    int kbpc = p.kb_per_chunk, nch = p.nchunks;
    if (I8 && warp >= 1 && p.bound_a && p.bound_b) {
        if (warp == 2 || warp == 3) {
            const unsigned* hdr = warp == 2 ? p.bound_a : p.bound_b;
            const unsigned h = hdr[0];
            const int np = min(static_cast<int>(h & kBoundCountMask), kBoundSlots - 1);
            unsigned m = 0u;
            for (int i = lane; i < np; i += 32) m = max(m, hdr[1 + i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) {
                const unsigned mult = (h & kBoundRowNorms) ? 1u
                                      : static_cast<unsigned>(warp == 2 ? p.row_chunks_a : p.row_chunks_b);
                // 0: no bound recorded (the staging took the plain kernel)
                bound_max[warp - 2] = np > 0 ? m : 0xFFFFFFFFu;
                bound_max[warp] = mult;
            }
        }
        named_barrier_sync(1, 32 * (1 + Cfg::EPI_WARPS));
        if (bound_max[0] != 0xFFFFFFFFu && bound_max[1] != 0xFFFFFFFFu) {
            const unsigned long long a2 = static_cast<unsigned long long>(bound_max[2]) * bound_max[0];
            const unsigned long long b2 = static_cast<unsigned long long>(bound_max[3]) * bound_max[1];
            // a2 * b2 < 2^48, without overflow (a2, b2 < 2^40)
            if (a2 == 0 || b2 <= ((1ull << 48) - 1) / a2) {
                kbpc = p.nkb;
                nch = 1;
            }
        }
    }

    const GemmCta c{smem, epi_stage, full, empty, tfull, tempty, drain, abort_flag, tmem_base,
                    rank, leader, cta_unit, num_units, total, total0};
    bool arrived = false;
    if (warp == 0) gemm_producer<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI, GRP>(tmA, tmB, P, c);
    else if (warp == 1) gemm_mma<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI, GRP>(P, c, kbpc, nch);
    else arrived = gemm_epilogue<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI, GRP>(tmC, P, c, nch);

    tc_fence_before();
    if (PAIR && !arrived) {
        // The producer and the MMA issuer arrive as soon as their roles end.
        // The barrier completes once every epilogue warp of both CTAs has
        // read its last accumulator, which it does only after the MMAs into
        // its TMEM completed: then the leader's MMAs into the peer's TMEM are
        // done and TMEM can be released.
        __syncwarp();
        cluster_arrive();
    }
    __syncthreads();
    if (PAIR) {
        __syncwarp();
        cluster_wait();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    if (p.clk && threadIdx.x == 0 && static_cast<int>(blockIdx.x) < p.clk_cap) {
        pdl_wait();
        const unsigned long long clk1 = clock64();
        const unsigned long long ns1 = global_ns_ordered();
        unsigned long long* r = p.clk + 4 * static_cast<int64_t>(blockIdx.x);
        r[0] = clk0;
        r[1] = clk1;
        r[2] = ns0;
        r[3] = ns1;
    }
}

template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI>
__global__ void __launch_bounds__(GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    const int total = p.mt * p.nt * p.batch;
    gemm_body<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI, false>(&tmA, &tmB, &tmC, &p, total, total);
}

// Two independent FP8 GEMMs (bf16 outputs) in one launch of single CTAs:
// each problem keeps its own operand layouts, steps, output and raster.
struct GemmGroup {
    CUtensorMap tmA[2], tmB[2], tmC[2];
    GemmParams p[2];
    int total0, total;
};

template <int BN, bool WIDE_EPI>
__global__ void __launch_bounds__(GemmCfg<BN, false, false, false, false, WIDE_EPI>::THREADS, 1)
    gemm_tc_group_kernel(const __grid_constant__ GemmGroup g) {
    gemm_body<BN, false, false, false, false, WIDE_EPI, true>(g.tmA, g.tmB, g.tmC, g.p, g.total0,
                                                               g.total);
}

// ====================================================================== host
// Per-device diagnostic buffers for the GEMM clock records (sq_set_clock_probe).
struct ClockProbe {
    std::atomic<unsigned long long*> fp8{nullptr};
    std::atomic<unsigned long long*> i8{nullptr};
    std::atomic<int> cap{0};
};
static ClockProbe g_clock_probe[64];

static ClockProbe* current_probe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    return &g_clock_probe[dev];
}

cudaError_t set_gemm_clock_probe(unsigned long long* fp8, unsigned long long* i8, int cap) {
    ClockProbe* cp = current_probe();
    if (!cp) return cudaErrorInvalidDevice;
    cp->cap.store(cap);
    cp->fp8.store(fp8);
    cp->i8.store(i8);
    return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major [outer, inner] (inner contiguous, row pitch `pitch` bytes), tiles
// of box_inner x box_outer elements, 128-byte swizzle, zero fill outside.
static bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                      uint64_t outer, uint64_t pitch, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Used for the INT8 path's fp16 operands; no L2 promotion measured ~1% faster
// there than 256-byte promotion.
static bool encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                      uint64_t rows, uint64_t batch, uint64_t pitch, uint64_t bpitch,
                      uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {pitch, bpitch};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool I8, bool A_MN, bool B_MN, bool PAIR, bool WIDE_EPI>
static cudaError_t run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                            const GemmParams& p, cudaStream_t st, int sms) {
    using Cfg = GemmCfg<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    auto kern = gemm_tc_kernel<BN, I8, A_MN, B_MN, PAIR, WIDE_EPI>;
    // CTAs (or CTA pairs) that fit this device at once
    const std::pair<cudaError_t, int> fit = per_device_once(reinterpret_cast<const void*>(kern), [&] {
        cudaError_t attr_err =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        int max_units = 0;
        if (attr_err != cudaSuccess) return std::make_pair(attr_err, 0);
        if (PAIR) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
            cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
            cfg.dynamicSmemBytes = Cfg::SMEM;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            attr_err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            max_units = n;
        } else {
            max_units = sms;
        }
        if (attr_err == cudaSuccess && max_units < 1) attr_err = cudaErrorInvalidConfiguration;
        return std::make_pair(attr_err, max_units);
    });
    if (fit.first != cudaSuccess) return fit.first;
    const int max_units = fit.second;
    const int total = p.mt * p.nt * p.batch;
    const int units = total < max_units ? total : max_units;
    if (!PAIR) return launch_pdl(kern, dim3(units), dim3(Cfg::THREADS), Cfg::SMEM, st, 1u, ta, tb, tc, p);
    return launch_pdl(kern, dim3(2 * units), dim3(Cfg::THREADS), Cfg::SMEM, st, 2u, ta, tb, tc, p);
}

// Tile shape: 256 x 256 on CTA pairs when there are enough such tiles to give
// every pair of SMs work, else 128 x 256 or 128 x 128 on single CTAs.
enum class Shape { Pair256, Single256, Single128 };

static Shape pick_shape(int64_t M, int64_t N, int64_t batch, int sms) {
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256) * batch;
    const int64_t wide_tiles = ((M + 127) / 128) * ((N + 255) / 256) * batch;
    if (pair_tiles >= sms / 2) return Shape::Pair256;
    if (wide_tiles >= sms) return Shape::Single256;
    return Shape::Single128;
}

// One FP8 problem's operand maps (A in boxes of 128 rows; B in boxes of b_rows
// rows, or of 128 columns when it is N-major) and, where its bf16 rows are
// 16-byte multiples, the map of the 32 x 32 output boxes; sets p.mt, p.nt,
// p.idesc and p.tma_store for tiles of tile_m x bn.
static bool fp8_problem_maps(const uint8_t* A, const uint8_t* B, int M, int N, int K, bool a_mn,
                             bool b_mn, int tile_m, int bn, int b_rows, int fmt, GemmParams& p,
                             CUtensorMap* ta, CUtensorMap* tb, CUtensorMap* tc) {
    bool ok;
    if (a_mn) ok = encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, M, K, M, 128, kBKBytes);
    else ok = encode_2d(ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, kBKBytes, kBM);
    if (!ok) return false;
    if (b_mn) ok = encode_2d(tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, N, K, N, 128, kBKBytes);
    else ok = encode_2d(tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, kBKBytes, b_rows);
    if (!ok) return false;
    p.mt = (M + tile_m - 1) / tile_m;
    p.nt = (N + bn - 1) / bn;
    p.idesc = idesc_make(static_cast<uint32_t>(fmt), static_cast<uint32_t>(fmt), a_mn, b_mn,
                         static_cast<uint32_t>(tile_m), static_cast<uint32_t>(bn));
    memset(tc, 0, sizeof(*tc));
    p.tma_store = 0;
    if (!p.out_e4m3 && N % 8 == 0 && reinterpret_cast<uintptr_t>(p.C) % 16 == 0) {
        if (!encode_2d(tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.C, N, M, static_cast<uint64_t>(N) * 2,
                       32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return false;
        p.tma_store = 1;
    }
    return true;
}

template <bool A_MN, bool B_MN, int BN, bool PAIR>
static cudaError_t gemm_fp8_shape(const uint8_t* A, const uint8_t* B, int M, int N, int K,
                                  GemmParams p, int fmt, cudaStream_t st, int sms) {
    using Cfg = GemmCfg<BN, false, A_MN, B_MN, PAIR, false>;   // tile geometry only
    CUtensorMap ta, tb, tc;
    if (!fp8_problem_maps(A, B, M, N, K, A_MN, B_MN, Cfg::TILE_M, BN, Cfg::B_ROWS, fmt, p, &ta, &tb,
                          &tc))
        return cudaErrorInvalidValue;
    // one round of 256-wide tiles leaves the epilogue exposed: give it 8 warps
    if (BN == 256 && static_cast<int64_t>(p.mt) * p.nt <= (PAIR ? sms / 2 : sms))
        return run_gemm<BN, false, A_MN, B_MN, PAIR, true>(ta, tb, tc, p, st, sms);
    return run_gemm<BN, false, A_MN, B_MN, PAIR, false>(ta, tb, tc, p, st, sms);
}

// FP8 tile shape by estimated time: rounds of tiles over the SMs (or SM
// pairs) times the k-blocks per tile times the time of one k-block on one SM,
// in clocks, plus a fixed cost for CTA pairs.  A k-block is 128 bytes of K.
// The per-k-block times are those the large workload measured on GB300 with
// every SM busy: 454 clk for a 128 x 128 tile, 784 for 128 x 256, 702 for
// each CTA's 128 x 256 half of a 256 x 256 pair tile.  The pair's fixed cost
// (~4000 clk) is its set-up (pair TMEM allocation, cluster barrier) and its
// longer exposed epilogue, measured on one-round launches: there 256 x 256
// pairs lost to single CTAs despite the shorter K loop.  Ties go to the later
// entry of the list.
static Shape pick_shape_fp8(int64_t M, int64_t N, int64_t K, int sms, int64_t* est = nullptr) {
    struct Cand { Shape s; int64_t tm, tn, slots, clk, fixed; };
    const Cand c[3] = {{Shape::Single256, 128, 256, sms, 784, 0},
                       {Shape::Single128, 128, 128, sms, 454, 0},
                       {Shape::Pair256, 256, 256, sms / 2, 702, 4000}};
    const int64_t nkb = (K + kBKBytes - 1) / kBKBytes;
    Shape best = Shape::Single128;
    int64_t best_t = -1;
    for (const Cand& x : c) {
        const int64_t tiles = ((M + x.tm - 1) / x.tm) * ((N + x.tn - 1) / x.tn);
        const int64_t rounds = (tiles + x.slots - 1) / x.slots;
        const int64_t t = rounds * nkb * x.clk + x.fixed;
        if (best_t < 0 || t <= best_t) {
            best = x.s;
            best_t = t;
        }
    }
    if (est) *est = best_t;
    return best;
}

template <bool A_MN, bool B_MN>
static cudaError_t gemm_fp8_layout(const uint8_t* A, const uint8_t* B, int M, int N, int K,
                                   const GemmParams& p, int fmt, cudaStream_t st, int sms) {
    switch (pick_shape_fp8(M, N, K, sms)) {
        case Shape::Pair256: return gemm_fp8_shape<A_MN, B_MN, 256, true>(A, B, M, N, K, p, fmt, st, sms);
        case Shape::Single256: return gemm_fp8_shape<A_MN, B_MN, 256, false>(A, B, M, N, K, p, fmt, st, sms);
        default: return gemm_fp8_shape<A_MN, B_MN, 128, false>(A, B, M, N, K, p, fmt, st, sms);
    }
}

cudaError_t launch_gemm_fp8(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            int fmt, int layout, int M, int N, int K, void* C,
                            const float* out_scale, const float* bias, unsigned* err_word,
                            cudaStream_t st, int sms) {
    GemmParams p{};
    p.bias = bias;
    p.M = M; p.N = N; p.K = K; p.batch = 1;
    p.nkb = (K + kBKBytes - 1) / kBKBytes;
    p.kb_per_chunk = p.nkb;
    p.nchunks = 1;
    p.sa = sa; p.sb = sb; p.C = C; p.acc_out = nullptr; p.strideC = 0;
    p.out_scale = out_scale;
    p.out_e4m3 = out_scale != nullptr;
    p.group_m = kGroupM;
    p.ga = p.gb = 1;
    p.Mg = M; p.Ng = N;
    // 16-byte stores: 8 bf16 or 16 E4M3 codes per row piece
    p.vec_store = (N % (p.out_e4m3 ? 16 : 8) == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0);
    p.err_word = err_word;
    if (ClockProbe* cp = current_probe()) {
        p.clk = cp->fp8.load();
        p.clk_cap = p.clk ? cp->cap.load() : 0;
    }
    if (layout == 0) return gemm_fp8_layout<false, false>(A, B, M, N, K, p, fmt, st, sms);
    if (layout == 1) return gemm_fp8_layout<false, true>(A, B, M, N, K, p, fmt, st, sms);
    return gemm_fp8_layout<true, true>(A, B, M, N, K, p, fmt, st, sms);
}

// ------------------------------------------------------------- grouped FP8
// Makespan, in clocks, of a grouped launch of tile_m x bn tiles: each tile of
// problem i costs its k-blocks times clk_kb, and the units are dealt to
// min(units, sms) CTAs in rounds of alternating direction, as unit_of deals
// them.
static int64_t group_makespan(const Fp8Problem* q, int bn, int64_t clk_kb, int sms) {
    int64_t tiles[2], cost[2];
    for (int i = 0; i < 2; ++i) {
        tiles[i] = static_cast<int64_t>((q[i].M + kBM - 1) / kBM) * ((q[i].N + bn - 1) / bn);
        cost[i] = static_cast<int64_t>((q[i].K + kBKBytes - 1) / kBKBytes) * clk_kb;
    }
    const int64_t total = tiles[0] + tiles[1];
    const int64_t g = total < sms ? total : sms;
    std::vector<int64_t> load(static_cast<size_t>(g), 0);
    for (int64_t u = 0; u < total; ++u) {
        const int64_t r = u / g, j = u % g;
        load[static_cast<size_t>((r & 1) ? g - 1 - j : j)] += u < tiles[0] ? cost[0] : cost[1];
    }
    int64_t m = 0;
    for (int64_t v : load) m = v > m ? v : m;
    return m;
}

template <int BN, bool WIDE_EPI>
static cudaError_t run_gemm_group(const Fp8Problem* q, int fmt, unsigned* err_word,
                                  cudaStream_t st, int sms) {
    using Cfg = GemmCfg<BN, false, false, false, false, WIDE_EPI>;
    auto kern = gemm_tc_group_kernel<BN, WIDE_EPI>;
    const cudaError_t attr = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), Cfg::SMEM);
    if (attr != cudaSuccess) return attr;
    GemmGroup g;
    memset(&g, 0, sizeof(g));
    ClockProbe* cp = current_probe();
    for (int i = 0; i < 2; ++i) {
        GemmParams& p = g.p[i];
        p.M = q[i].M; p.N = q[i].N; p.K = q[i].K; p.batch = 1;
        p.nkb = (q[i].K + kBKBytes - 1) / kBKBytes;
        p.kb_per_chunk = p.nkb;
        p.nchunks = 1;
        p.sa = q[i].sa; p.sb = q[i].sb; p.C = q[i].C;
        p.group_m = kGroupM;
        p.ga = p.gb = 1;
        p.Mg = q[i].M; p.Ng = q[i].N;
        p.vec_store = (q[i].N % 8 == 0) && (reinterpret_cast<uintptr_t>(q[i].C) % 16 == 0);
        p.err_word = err_word;
        p.a_mn = q[i].layout == 2;
        p.b_mn = q[i].layout != 0;
        if (cp) {
            p.clk = cp->fp8.load();
            p.clk_cap = p.clk ? cp->cap.load() : 0;
        }
        if (!fp8_problem_maps(q[i].A, q[i].B, q[i].M, q[i].N, q[i].K, p.a_mn != 0, p.b_mn != 0, kBM,
                              BN, BN, fmt, p, &g.tmA[i], &g.tmB[i], &g.tmC[i]))
            return cudaErrorInvalidValue;
    }
    g.total0 = g.p[0].mt * g.p[0].nt;
    g.total = g.total0 + g.p[1].mt * g.p[1].nt;
    const int units = g.total < sms ? g.total : sms;
    return launch_pdl(kern, dim3(units), dim3(Cfg::THREADS), Cfg::SMEM, st, 1u, g);
}

// Grouped when the estimate says one launch of both beats two launches: the
// group's makespan (plus the last tile's exposed epilogue, ~0.9 us on 128-wide
// tiles and ~1.7 us on 256-wide ones) against the two launches' estimates
// plus the second launch's ramp (its CTAs start only as the first launch's
// leave, then set up and wait for their first operands: ~2.5 us measured).
// Only groups of at most four rounds of tiles are considered: larger
// problems keep their own launches and CTA-pair tiles.
cudaError_t launch_gemm_fp8_pair(const Fp8Problem* q, int fmt, unsigned* err_word, cudaStream_t st,
                                 int sms) {
    int64_t sep = 5000;
    for (int i = 0; i < 2; ++i) {
        int64_t e = 0;
        pick_shape_fp8(q[i].M, q[i].N, q[i].K, sms, &e);
        sep += e;
    }
    auto units = [&](int bn) {
        int64_t u = 0;
        for (int i = 0; i < 2; ++i)
            u += static_cast<int64_t>((q[i].M + kBM - 1) / kBM) * ((q[i].N + bn - 1) / bn);
        return u;
    };
    const int64_t cap = 4 * static_cast<int64_t>(sms);
    const int64_t g128 = units(128) <= cap ? group_makespan(q, 128, 454, sms) + 1800 : INT64_MAX;
    const int64_t g256 = units(256) <= cap ? group_makespan(q, 256, 784, sms) + 3400 : INT64_MAX;
    if (g256 < sep && g256 <= g128) return run_gemm_group<256, true>(q, fmt, err_word, st, sms);
    if (g128 < sep) return run_gemm_group<128, false>(q, fmt, err_word, st, sms);
    for (int i = 0; i < 2; ++i) {
        const cudaError_t e = launch_gemm_fp8(q[i].A, q[i].B, q[i].sa, q[i].sb, fmt, q[i].layout,
                                              q[i].M, q[i].N, q[i].K, q[i].C, nullptr, nullptr,
                                              err_word, st, sms);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int BN, bool PAIR>
static cudaError_t gemm_i8_shape(const uint16_t* A16, const uint16_t* B16, int batch, int M, int N,
                                 int K, GemmParams p, cudaStream_t st, int sms) {
    using Cfg = GemmCfg<BN, true, false, false, PAIR, false>;
    const int bk = kBKBytes / 2;   // 64 fp16 per k-block
    CUtensorMap ta, tb;
    if (!encode_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A16, K, M, batch,
                   static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(M) * K * 2, bk, kBM))
        return cudaErrorInvalidValue;
    if (!encode_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B16, K, N, batch,
                   static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(N) * K * 2, bk, Cfg::B_ROWS))
        return cudaErrorInvalidValue;
    p.mt = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
    p.nt = (N + BN - 1) / BN;
    p.idesc = idesc_make(0, 0, false, false, Cfg::TILE_M, BN);   // F16 x F16 -> F32
    // The INT8 epilogue stores from the threads: TMA stores of its fp32 boxes
    // (twice the bytes of the FP8 output, from 8 warps) measured 17% slower on
    // the large workload, competing with the operand loads for the TMA unit.
    CUtensorMap tc;
    memset(&tc, 0, sizeof(tc));
    p.tma_store = 0;
    return run_gemm<BN, true, false, false, PAIR, false>(ta, tb, tc, p, st, sms);
}

cudaError_t launch_gemm_i8(const uint16_t* A16, const uint16_t* B16, const float* sA,
                           const float* sB, int ga, int gb, int batch, int M, int N, int K,
                           int64_t strideC, float* C, int32_t* acc_out, const unsigned* bound_a,
                           const unsigned* bound_b, unsigned* err_word, cudaStream_t st, int sms) {
    const int bk = kBKBytes / 2;
    GemmParams p{};
    p.M = M; p.N = N; p.K = K; p.batch = batch;
    p.group_m = kGroupMI8;
    p.nkb = (K + bk - 1) / bk;
    p.kb_per_chunk = kI8ChunkK / bk;
    p.nchunks = (p.nkb + p.kb_per_chunk - 1) / p.kb_per_chunk;
    p.sa = sA; p.sb = sB; p.C = C; p.acc_out = acc_out; p.strideC = strideC;
    p.ga = ga; p.gb = gb;
    p.Mg = (M + ga - 1) / ga;
    p.Ng = (N + gb - 1) / gb;
    p.vec_store = (N % 4 == 0) && (strideC % 4 == 0) &&
                  (reinterpret_cast<uintptr_t>(C) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(acc_out) % 16 == 0);
    p.sb_vec = (gb == 1) && (N % 4 == 0) && (reinterpret_cast<uintptr_t>(sB) % 16 == 0);
    p.err_word = err_word;
    if (ClockProbe* cp = current_probe()) {
        p.clk = cp->i8.load();
        p.clk_cap = p.clk ? cp->cap.load() : 0;
    }
    p.bound_a = bound_a;
    p.bound_b = bound_b;
    // a row of K codes overlaps at most ceil(K / chunk) + 1 staged chunks
    p.row_chunks_a = p.row_chunks_b = (K + kStgChunk - 1) / kStgChunk + 1;
    if (pick_shape(M, N, batch, sms) == Shape::Pair256)
        return gemm_i8_shape<256, true>(A16, B16, batch, M, N, K, p, st, sms);
    // Very small problems (fewer 128 x 256 tiles than a quarter of the SMs)
    // spread over 128 x 128 tiles: measured 17-25% faster there, 6-10%
    // slower than 128 x 256 tiles once those fill a good part of the GPU.
    const int64_t wide_tiles = ((M + 127) / 128) * ((N + 255) / 256) * static_cast<int64_t>(batch);
    if (wide_tiles < sms / 4) {
        // When even 128 x 64 (or 128 x 32) tiles make one round, take those:
        // each CTA then streams a half (a quarter) of the B rows and stores
        // that share of the outputs, which bound these few-CTA launches per
        // SM, at the cost of reading A more often over more SMs.
        const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128) * static_cast<int64_t>(batch);
        if (4 * tiles <= sms) return gemm_i8_shape<32, false>(A16, B16, batch, M, N, K, p, st, sms);
        if (2 * tiles <= sms) return gemm_i8_shape<64, false>(A16, B16, batch, M, N, K, p, st, sms);
        return gemm_i8_shape<128, false>(A16, B16, batch, M, N, K, p, st, sms);
    }
    return gemm_i8_shape<256, false>(A16, B16, batch, M, N, K, p, st, sms);
}

// ---------------------------------------------------------------- staging
// Small or strided operands: a grid-stride kernel over up to two staging
// jobs at once (A and B of one GEMM call share the launch).
struct StageJob {
    const int8_t* src;
    int64_t rows, K, stride;    // rows per batch; batch b starts at src + b*stride
    int64_t total;              // 16-code pieces: batch * rows * K / 16
    uint16_t* dst;
    unsigned* bound;            // the operand's bound header (nullable): set to "none"
};

__global__ void __launch_bounds__(256) i8_to_f16_kernel(const StageJob j0, const StageJob j1) {
    pdl_begin();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (j0.bound) *j0.bound = 0u;   // this path records no bound
        if (j1.bound) *j1.bound = 0u;
    }
    // 16 codes per step: one 16-B load, two 16-B stores (K % 16 == 0)
    const int64_t all = j0.total + j1.total;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < all;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool first = u < j0.total;
        const StageJob& j = first ? j0 : j1;
        const int64_t v = first ? u : u - j0.total;
        const int64_t per_batch = j.rows * (j.K / 16);
        const int64_t b = v / per_batch;
        const int64_t r = v - b * per_batch;
        const uint4 raw = ld_stream_v4(j.src + b * j.stride + r * 16);
        uint16_t* d = j.dst + v * 16;
        st_v4(d, i8x8_to_f16x8(make_uint2(raw.x, raw.y)));
        st_v4(d + 8, i8x8_to_f16x8(make_uint2(raw.z, raw.w)));
    }
}

// Contiguous source (batch stride == rows*K): a bulk-copy pipeline per warp,
// as in the FP8 quantize.  Every warp of a persistent CTA streams its own
// chunks of kStgChunk codes (1 KB in, 2 KB of fp16 out) through a kStgStages-
// deep ring with bulk copies and its own mbarriers; lane 0 waits and issues,
// a warp barrier orders the other lanes, and no CTA-wide barrier is needed
// inside the loop.  Each lane converts four 8-byte pieces (conflict-free
// shared-memory access).  The ragged tail (a multiple of 16 codes, below one
// chunk) is done by block 0 with vector loads.
constexpr int kStgWarps = 24;
constexpr int kStgStages = 2;
constexpr int kStgWarpBytes = kStgStages * kStgChunk + 2 * kStgChunk * 2;
constexpr int kStgSmem = kStgWarps * kStgWarpBytes + kStgWarps * kStgStages * 8 + 128;

__global__ void __launch_bounds__(kStgWarps * 32) i8_to_f16_bulk_kernel(const int8_t* __restrict__ src,
                                                                       int64_t n,
                                                                       uint16_t* __restrict__ dst,
                                                                       unsigned* __restrict__ bound,
                                                                       unsigned* err_word) {
    extern __shared__ uint8_t gsmem_raw[];
    uint8_t* gsmem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(gsmem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* in_buf = gsmem + warp * kStgWarpBytes;              // kStgStages x 1 KB
    uint8_t* out_buf = in_buf + kStgStages * kStgChunk;          // 2 x 2 KB
    uint64_t* full = reinterpret_cast<uint64_t*>(gsmem + kStgWarps * kStgWarpBytes) + warp * kStgStages;
    __shared__ int abort_flag;
    __shared__ unsigned warp_max[kStgWarps];
    __shared__ unsigned tail_sq;
    unsigned chunk_max = 0u;       // largest sum of squared codes over this warp's chunks
    const int64_t nfull = n / kStgChunk;
    const int64_t GW = static_cast<int64_t>(gridDim.x) * kStgWarps;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * kStgWarps + warp;
    const int64_t count = gw < nfull ? (nfull - gw + GW - 1) / GW : 0;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        tail_sq = 0u;
    }
    if (lane == 0) {
        for (int k = 0; k < kStgStages; ++k) mbar_init(&full[k], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing above touches global memory (it overlaps the previous kernel)
    pdl_begin();
    if (lane == 0) {
        for (int64_t k = 0; k < count && k < kStgStages; ++k) {
            mbar_arrive_expect_tx(&full[k], kStgChunk);
            bulk_load(in_buf + k * kStgChunk, src + (gw + k * GW) * kStgChunk, kStgChunk, &full[k]);
        }
    }
    int64_t i = 0;
    for (; i < count; ++i) {
        const int stage = static_cast<int>(i % kStgStages);
        const int ob = static_cast<int>(i & 1);
        int ok = 1;
        if (lane == 0) {
            ok = mbar_wait(&full[stage], static_cast<uint32_t>((i / kStgStages) & 1), &abort_flag, err_word);
            if (i >= 2) bulk_wait_read<1>();   // the store from out_buf[ob] two chunks ago is read
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();                          // orders lane 0's wait before the other lanes' reads
        if (!ok) break;
        const uint8_t* in = in_buf + stage * kStgChunk;
        uint8_t* out = out_buf + ob * kStgChunk * 2;
        uint2 w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = *reinterpret_cast<const uint2*>(in + (k * 32 + lane) * 8);
#pragma unroll
        for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(out + (k * 32 + lane) * 16) = i8x8_to_f16x8(w[k]);
        int sq = 0;                // sum of squares of this lane's 32 codes (<= 32 * 127^2)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sq = __dp4a(static_cast<int>(w[k].x), static_cast<int>(w[k].x), sq);
            sq = __dp4a(static_cast<int>(w[k].y), static_cast<int>(w[k].y), sq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        chunk_max = max(chunk_max, static_cast<unsigned>(sq));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            const int64_t c = gw + i * GW;
            bulk_store(dst + c * kStgChunk, out, kStgChunk * 2);
            bulk_commit();
            if (i + kStgStages < count) {
                mbar_arrive_expect_tx(&full[stage], kStgChunk);
                bulk_load(in_buf + stage * kStgChunk, src + (c + kStgStages * GW) * kStgChunk, kStgChunk,
                          &full[stage]);
            }
        }
    }
    if (lane == 0) {
        if (i < count) {
            // gave up on a wait: let the loads already issued land before exiting
            for (int64_t j = i; j < count && j < i + kStgStages; ++j)
                mbar_wait_drain(&full[j % kStgStages], static_cast<uint32_t>((j / kStgStages) & 1));
        }
        bulk_wait_all();
    }
    if (lane == 0) warp_max[warp] = chunk_max;
    if (blockIdx.x == 0) {
        // the ragged tail (< one chunk) counts as one more chunk
        int tq = 0;
        for (int64_t e = nfull * kStgChunk + threadIdx.x * 8; e < n; e += kStgWarps * 32 * 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(src + e);
            *reinterpret_cast<uint4*>(dst + e) = i8x8_to_f16x8(v);
            tq = __dp4a(static_cast<int>(v.x), static_cast<int>(v.x), tq);
            tq = __dp4a(static_cast<int>(v.y), static_cast<int>(v.y), tq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tq += __shfl_xor_sync(0xffffffffu, tq, o);
        if (lane == 0 && tq != 0) atomicAdd(&tail_sq, static_cast<unsigned>(tq));
    }
    __syncthreads();
    if (threadIdx.x == 0 && bound) {
        unsigned m = tail_sq;
        for (int w = 0; w < kStgWarps; ++w) m = max(m, warp_max[w]);
        bound[1 + blockIdx.x] = m;
        if (blockIdx.x == 0) bound[0] = gridDim.x;   // slot count; chunk sums
    }
}

// CTAs of the bulk pipeline for one operand (one bound slot each), or 0 when
// the operand takes the plain kernel: contiguous operands of at least about
// 8192 codes per SM take the pipeline; smaller ones the plain kernel, with no
// large shared-memory carveout.
static int i8_staging_blocks(int64_t batch, int64_t rows, int64_t K, int64_t stride, int sms) {
    const int64_t n = batch * rows * K;
    if (!(stride == rows * K || batch == 1) || n < static_cast<int64_t>(8192) * sms) return 0;
    int64_t blocks = (n / kStgChunk + kStgWarps - 1) / kStgWarps;
    int64_t cap = static_cast<int64_t>(sms);
    if (cap > kStgMaxParts) cap = kStgMaxParts;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

// One operand through the bulk pipeline, when it qualifies.  Returns false if
// it does not.
static bool stage_bulk(const int8_t* src, int64_t batch, int64_t rows, int64_t K, int64_t stride,
                       uint16_t* dst, unsigned* bound, unsigned* err_word, cudaStream_t st,
                       int sms, cudaError_t* err) {
    const int blocks = i8_staging_blocks(batch, rows, K, stride, sms);
    if (!err_word || blocks == 0) return false;
    const int64_t n = batch * rows * K;
    const cudaError_t attr =
        set_max_dynamic_smem(reinterpret_cast<const void*>(i8_to_f16_bulk_kernel), kStgSmem);
    if (attr != cudaSuccess) {
        *err = attr;
        return true;
    }
    *err = launch_pdl(i8_to_f16_bulk_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kStgWarps * 32),
                      kStgSmem, st, 1u, src, n, dst, bound, err_word);
    return true;
}

static cudaError_t stage_plain(StageJob j0, StageJob j1, cudaStream_t st, int sms) {
    const int64_t all = j0.total + j1.total;
    int64_t blocks = (all + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(i8_to_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, 1u,
                      j0, j1);
}

cudaError_t launch_i8_to_f16_pair(const int8_t* a, int64_t M, const int8_t* b, int64_t N,
                                  int64_t batch, int64_t K, int64_t stride_a, int64_t stride_b,
                                  uint16_t* a16, uint16_t* b16, unsigned* bound_a,
                                  unsigned* bound_b, unsigned* err_word, cudaStream_t st,
                                  int sms) {
    StageJob small[2];
    int nsmall = 0;
    cudaError_t e = cudaSuccess;
    // B first: in the usual order of calls (quantize A, quantize B, GEMM) its
    // codes were written last and are the ones still in L2
    if (!stage_bulk(b, batch, N, K, stride_b, b16, bound_b, err_word, st, sms, &e))
        small[nsmall++] = StageJob{b, N, K, stride_b, batch * N * (K / 16), b16, bound_b};
    if (e != cudaSuccess) return e;
    if (!stage_bulk(a, batch, M, K, stride_a, a16, bound_a, err_word, st, sms, &e))
        small[nsmall++] = StageJob{a, M, K, stride_a, batch * M * (K / 16), a16, bound_a};
    if (e != cudaSuccess) return e;
    if (nsmall == 0) return cudaSuccess;
    if (nsmall == 1) small[1] = StageJob{nullptr, 1, 16, 0, 0, nullptr, nullptr};
    return stage_plain(small[0], small[1], st, sms);
}

cudaError_t launch_i8_to_f16_one(const int8_t* src, int64_t batch, int64_t rows, int64_t K,
                                 int64_t stride, uint16_t* dst, unsigned* bound,
                                 unsigned* err_word, cudaStream_t st, int sms) {
    cudaError_t e = cudaSuccess;
    if (stage_bulk(src, batch, rows, K, stride, dst, bound, err_word, st, sms, &e)) return e;
    return stage_plain(StageJob{src, rows, K, stride, batch * rows * (K / 16), dst, bound},
                       StageJob{nullptr, 1, 16, 0, 0, nullptr, nullptr}, st, sms);
}

}  // namespace sq
