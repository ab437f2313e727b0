// Grouped FP8 (e4m3) expert GEMMs with 128x128 block scales on tcgen05.
//
// "GPT-OSS on Day 0" (perplexity.ai hub blog) serves the experts as FP8 with
// 128x128 block scales on DeepGEMM, with the bias loaded into the
// accumulators once per output block; this is the sm_103a counterpart:
//
//   acc[r, n] = bias[n] + sum_kb (sa[r, kb] * sw[n/128, kb]) * P_kb[r, n],
//   P_kb      = sum_{k in block kb} a[r, k] * w[n, k]      (one 128-wide K block)
//
// tcgen05.mma (kind::f8f6f4) has no per-block fp32 scale, so each K block is
// accumulated on its own into a TMEM buffer (ping-pong), and the epilogue
// warps "promote" it into fp32 registers that started at the bias.
//
// Roles (one CTA per SM, persistent over a static tile list ordered expert,
// n-tile, m-tile so that the m-tiles of one weight tile run side by side and
// share it through L2):
//   warp 0      TMA producer: A (activation rows of one expert) and B (the
//               expert's weight rows) per K block into a STAGES-deep ring.
//   warp 1      TMEM allocator and MMA issuer (one thread): 4 MMAs of K=32
//               per K block into TMEM buffer kb % NBUF, then one commit to
//               the buffer's full barrier.  That commit also frees the K
//               block's smem stage: the first promotion warp releases the
//               stage when it sees the buffer full (one commit per K block
//               instead of two keeps the issuing thread on the MMAs).
//   warp 3      the second MMA issuer: warps 1 and 3 take alternate K blocks
//               (and so alternate TMEM buffers), each thread's waits and
//               issue overlapping the other's
//   warp 2      metadata: stages each tile's bias in shared memory one tile ahead
//   (warpgroup 0 gives registers to the promotion warpgroups)
//   warps 4-11  promotion + epilogue: tcgen05.ld the partial, FMA with the
//               two scales into registers, release the buffer; after the last
//               K block run the fused epilogue:
//                 gate/up GEMM: SwiGLU + 1x128 FP8 requant -> hq, sh
//                 down GEMM:    routing-weight scale -> part[t*k+j, :]
// Every mbarrier wait is bounded; a timeout sets an error bit and all roles
// drain and exit.
#include <cuda_bf16.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// Threads issuing the MMAs of one CTA (one per warp, warps 1 and 3 with two;
// two measured 1.2 % faster on a 16384-token, 4096-wide layer of 128 experts).
#ifndef MOE_PREFILL_MMA_ISSUERS
#define MOE_PREFILL_MMA_ISSUERS 2
#endif
constexpr int kMmaIssuers = MOE_PREFILL_MMA_ISSUERS;

template <bool GATED>
struct GemmCfg {
    static constexpr int BM = 128;
    // two 128-row weight blocks per tile, one N=256 MMA per K step: gate/up the
    // gate and the up block of one h block, down two consecutive w2 blocks
    static constexpr int BN = 256;
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 4;
    static constexpr int NBUF = 512 / BN;  // TMEM partial buffers (all 512 columns)
    static constexpr int EPI_WARPS = 8;                   // warpgroups 1 and 2
    static constexpr int THREADS = (4 + EPI_WARPS) * 32;  // warpgroup 0: producer, MMA, 2 idle warps
    // gate/up: the promotion warps hold 128 accumulators + 32 loaded columns, so
    // warpgroup 0 hands registers to them; the split must not ask for more than
    // it frees: 8*32*(200-168) = 8192 <= 4*32*(168-88) = 10240
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int WG0_REGS = 88;
    static constexpr int EPI_REGS = 200;
    static constexpr int COLS = BN / 2;  // accumulator columns per epilogue thread
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
    static constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
    static constexpr int HALVES = BN / 128;  // 128-column blocks of a tile (gate/up: gate and up)
};

struct TileInfo {
    int e, nt, row0, rows;
};

// Row block (of the expert's weight matrix) of a tile's block `which` (0/1):
// gate/up: the gate block and the up block of h block nt; down: blocks 2nt and
// 2nt+1, the second past the last one (== RB) when RB is odd -- it is then
// loaded as zeros or another expert's block and its results are dropped.
template <bool GATED>
__device__ __forceinline__ int weight_block(const GemmParams& p, int nt, int which) {
    return GATED ? (which ? p.up_rows / 128 + nt : nt) : 2 * nt + which;
}


__device__ __forceinline__ TileInfo decode_tile(int tile, const int* s_tiles, const int* s_off, const int* s_cnt,
                                                int E) {
    int lo = 0, hi = E;  // s_tiles[lo] <= tile < s_tiles[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= tile)
            lo = mid;
        else
            hi = mid;
    }
    TileInfo ti;
    ti.e = lo;
    const int local = tile - s_tiles[lo];
    const int mtc = (s_cnt[lo] + 127) >> 7;
    ti.nt = local / mtc;
    const int mt = local - ti.nt * mtc;
    ti.row0 = s_off[lo] + mt * 128;
    ti.rows = min(128, s_cnt[lo] - mt * 128);
    return ti;
}

template <bool GATED>
__global__ void __launch_bounds__(GemmCfg<GATED>::THREADS, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
    using C = GemmCfg<GATED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);

    __shared__ __align__(8) uint64_t full_bar[C::STAGES];
    __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[C::NBUF];
    __shared__ __align__(8) uint64_t tempty_bar[C::NBUF];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ __align__(8) uint64_t amax_bar;  // gate/up epilogue: the two column halves of a row meet here
    __shared__ __align__(8) uint64_t bfull_bar[2];   // bias slot filled by the metadata warp
    __shared__ __align__(8) uint64_t bempty_bar[2];  // bias slot read by every epilogue thread
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int s_tiles[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
    __shared__ float s_amax[2][2][128];  // [tile parity][column half][row]
    // staged one tile ahead by the metadata warp, per slot: the tile's bias, the
    // activation scales of its first two K blocks, the weight scales of those
    // K blocks (gate: [0..1], up: [2..3]), and for the down GEMM each row's
    // slot t*k+j and routing weight
    __shared__ float s_bias[2][C::BN];
    __shared__ float s_sa01[2][2][128];
    __shared__ float s_sw01[2][4];
    __shared__ int s_rslot[2][GATED ? 1 : 128];
    __shared__ float s_rw[2][GATED ? 1 : 128];
    // down GEMM: per epilogue warp, 32 rows x 16 fp32 (+4 pad: conflict-free
    // 16-byte accesses) that turn row-per-lane results into 64-byte row segments
    __shared__ __align__(16) float s_stage[GATED ? 1 : C::EPI_WARPS][32][20];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), C::EPI_WARPS);
        }
        mbar_init(smem_u32(&drain_bar), kMmaIssuers);
        mbar_init(smem_u32(&amax_bar), C::EPI_WARPS * 32);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bfull_bar[b]), 32);
            mbar_init(smem_u32(&bempty_bar[b]), C::EPI_WARPS * 32);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), 512);
    // Everything up to pdl_wait overlaps the previous kernel's tail.  The tile
    // lists come from the router's scan, which had completed before the kernel
    // ahead of this one let it be scheduled; read them from L2 now.
    for (int i = tid; i <= E; i += C::THREADS) {
        s_tiles[i] = __ldcg(p.tiles + i);
        s_off[i] = __ldcg(p.offset + i);
        if (i < E) s_cnt[i] = __ldcg(p.count + i);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    const int total = s_tiles[E];
    volatile int* abort_p = &abort_flag;
    uint32_t* err = p.status + kStatusError;
    // The weights are inputs of the layer: the producer fills the first
    // stages' weight boxes before waiting for the previous kernel, whose
    // output (the activation rows) it loads after the wait.
    int pre = 0;  // stages whose weight boxes are in flight before the wait
    if (warp == 0 && lane == 0) {
        for (int tile = blockIdx.x; tile < total && pre < C::STAGES; tile += gridDim.x) {
            const TileInfo ti = decode_tile(tile, s_tiles, s_off, s_cnt, E);
            const int blk0 = (ti.e * p.sw_rowblocks + weight_block<GATED>(p, ti.nt, 0)) * p.KB;
            const int blk1 = (ti.e * p.sw_rowblocks + weight_block<GATED>(p, ti.nt, 1)) * p.KB;
            for (int kb = 0; kb < p.KB && pre < C::STAGES; ++kb, ++pre) {
                const uint32_t fb = smem_u32(&full_bar[pre]);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                const uint32_t b_dst = smem_u32(smem + pre * C::STAGE_BYTES) + C::A_BYTES;
                tma_load_2d(b_dst, &tmB, 0, (blk0 + kb) * 128, fb);
                tma_load_2d(b_dst + 128 * 128, &tmB, 0, (blk1 + kb) * 128, fb);
            }
        }
    }
    // from here on this kernel reads what the previous kernels wrote
    pdl_wait();
    // No early launch_dependents: the next kernel starts when this grid
    // completes.  Releasing it here made the replayed qwen235b_prefill step
    // 93 us slower (oss120b_prefill 24 us), although its CTAs could only take
    // SMs as this grid's CTAs exit.

    if (warp < 4) {
        regs_release<C::WG0_REGS>();
    }
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0;  // bit s: stage s was filled at least once
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const TileInfo ti = decode_tile(tile, s_tiles, s_off, s_cnt, E);
                // blocked weights: block (e, row block, kb) starts at row ((e*RB + rb)*KB + kb)*128
                const int blk0 = (ti.e * p.sw_rowblocks + weight_block<GATED>(p, ti.nt, 0)) * p.KB;
                const int blk1 = (ti.e * p.sw_rowblocks + weight_block<GATED>(p, ti.nt, 1)) * p.KB;
                for (int kb = 0; kb < p.KB; ++kb) {
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    if (pre > 0) {
                        --pre;  // first use of this stage: its weights went out before the wait
                    } else {
                        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                        tma_load_2d(b_dst, &tmB, 0, (blk0 + kb) * 128, fb);
                        tma_load_2d(b_dst + 128 * 128, &tmB, 0, (blk1 + kb) * 128, fb);
                    }
                    tma_load_2d(a_dst, &tmA, kb * 128, ti.row0, fb);
                    filled |= 1u << stage;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: the last fill of every stage has landed (TMA completion
            // does not depend on the other roles) ...
            int dummy = 0;
            for (int i = 0; i < C::STAGES; ++i) {
                int s = (stage + C::STAGES - 1 - i) % C::STAGES;
                uint32_t ph = (s < stage) ? phase : phase ^ 1u;  // parity of that stage's last fill
                if (filled & (1u << s)) mbar_wait(smem_u32(&full_bar[s]), ph, &dummy, err, kErrTimeoutProducer);
            }
            // ... and, on the normal path, every stage was released by the
            // promotion warp, so no arrive can land after this CTA exits.
            if (ok) {
                for (int i = 0; i < C::STAGES; ++i) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1 || (kMmaIssuers == 2 && warp == 3)) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuers
            // With two issuers (warps 1 and 3), the CTA's K blocks alternate
            // between them: K block q of this CTA's sequence (tile after tile)
            // goes to issuer q % 2, always into TMEM buffer q % 2, so each
            // thread's per-K-block work (barrier waits, descriptors, MMA
            // issue, commit) has two K blocks' time.
            const int me = warp == 1 ? 0 : 1;
            bool ok = true;
            int q = 0;  // position in this CTA's K-block sequence
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                for (int kb = 0; kb < p.KB && ok; ++kb, ++q) {
                    if (q % kMmaIssuers != me) continue;
                    const int stage = q % C::STAGES, buf = q % C::NBUF;
                    const uint32_t sphase = (uint32_t)(q / C::STAGES) & 1u, tphase = (uint32_t)(q / C::NBUF) & 1u;
                    if (!mbar_wait(smem_u32(&full_bar[stage]), sphase, abort_p, err, kErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_base = a_base + C::A_BYTES;
                    // one N = BN MMA per K step (gate/up: the 128 gate and the 128 up
                    // weight rows are one 256-row B operand)
                    if (!mbar_wait(smem_u32(&tempty_bar[buf]), tphase ^ 1u, abort_p, err, kErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(buf * C::BN);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_e4m3(d, smem_desc_sw128(a_base + 32 * k4), smem_desc_sw128(b_base + 32 * k4), C::IDESC,
                                 k4 > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&tfull_bar[buf]));
                }
            }
            // every MMA issued above has completed before TMEM is released
            mma_commit(smem_u32(&drain_bar));
            int dummy = 0;
            mbar_wait(smem_u32(&drain_bar), 0, &dummy, err, kErrTimeoutMma);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------- metadata warp
        // Stages each tile's bias in shared memory one tile ahead, so the
        // epilogue warps never start a tile with a wait on global memory.
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(smem_u32(&bempty_bar[slot]), use ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
            const TileInfo t = decode_tile(tile, s_tiles, s_off, s_cnt, E);
            const uint16_t* bias_e = p.bias + (size_t)t.e * (GATED ? 2 * p.N_real : p.N_real);
            for (int c = lane; c < C::BN; c += 32) {
                // gate/up: h feature nt*128 + c%128 of the gate (c < 128) or up half of b13;
                // down: output feature (2nt + c/128)*128 + c%128
                const int n = (GATED ? t.nt : 2 * t.nt + (c >> 7)) * 128 + (c & 127);
                s_bias[slot][c] =
                    n < p.N_real ? bf16_bits_to_f32(__ldg(bias_e + (GATED ? (c >> 7) * p.N_real : 0) + n)) : 0.f;
            }
            for (int r = lane; r < 128; r += 32) {
                const int gr = min(t.row0 + r, p.R - 1);
                s_sa01[slot][0][r] = __ldg(p.sa + gr);
                s_sa01[slot][1][r] = p.KB > 1 ? __ldg(p.sa + (size_t)p.R + gr) : 0.f;
                if (!GATED) {
                    const int st = __ldg(p.perm + gr);
                    s_rslot[slot][r] = st;
                    s_rw[slot][r] = bf16_bits_to_f32(__ldg(p.topk_wb + st));
                }
            }
            if (lane < 4) {
                const int kb = lane & 1, which = lane >> 1;  // lanes: block 0 kb 0, 1; block 1 kb 0, 1
                const int b = weight_block<GATED>(p, t.nt, which);
                float v = 0.f;
                if (kb < p.KB && b < p.sw_rowblocks) v = __ldg(p.sw + ((size_t)t.e * p.sw_rowblocks + b) * p.KB + kb);
                s_sw01[slot][lane] = v;
            }
            mbar_arrive(smem_u32(&bfull_bar[slot]));
        }
    } else if (warp >= 4) {
        // -------------------------------------------- promotion + epilogue
        regs_acquire<C::EPI_REGS>();
        const int ew = warp - 4;
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int half = ew >> 2;      // which half of the columns
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int buf = 0;
        int e_stage = 0;
        uint32_t tphase = 0;
        uint32_t tpar = 0;  // parity of the tiles this CTA has finished
        bool ok = true;
        int tcount = 0;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, tpar ^= 1u, ++tcount) {
            const TileInfo ti = decode_tile(tile, s_tiles, s_off, s_cnt, E);
            const int grow = ti.row0 + row;
            const bool valid = row < ti.rows;
            const int grow_c = min(grow, p.R - 1);
            float acc[C::COLS];
            const int n0 = ti.nt * 128 + 64 * half;
            const int bslot = tpar;  // tiles alternate between the two bias slots
            const uint32_t buse = (uint32_t)(tcount >> 1) & 1u;
            if (!mbar_wait(smem_u32(&bfull_bar[bslot]), buse, abort_p, err, kErrTimeoutEpilogue)) break;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                acc[i] = s_bias[bslot][64 * half + i];
                acc[64 + i] = s_bias[bslot][128 + 64 * half + i];
            }
            // scales of K blocks 0 and 1 (later ones are loaded two K blocks ahead)
            float a0 = s_sa01[bslot][0][row], a1 = s_sa01[bslot][1][row];
            float g0 = s_sw01[bslot][0], g1 = s_sw01[bslot][1], u0 = s_sw01[bslot][2], u1 = s_sw01[bslot][3];
            const int my_slot = GATED ? 0 : s_rslot[bslot][GATED ? 0 : row];
            const float my_w = GATED ? 0.f : s_rw[bslot][GATED ? 0 : row];
            mbar_arrive(smem_u32(&bempty_bar[bslot]));
            const float* sa_row = p.sa + grow_c;  // element kb at sa_row[kb * R]
            const int b1 = weight_block<GATED>(p, ti.nt, 1);
            const bool has1 = b1 < p.sw_rowblocks;  // down GEMM, odd block count: the last tile has one block
            const float* sw0 = p.sw + ((size_t)ti.e * p.sw_rowblocks + weight_block<GATED>(p, ti.nt, 0)) * p.KB;
            const float* sw1 = p.sw + ((size_t)ti.e * p.sw_rowblocks + b1) * p.KB;
            // Warps whose TMEM lane quarter holds no valid row of this tile only
            // keep the buffer hand-over going (decode tiles have few rows).
            const bool active = quarter * 32 < ti.rows;
            // scales of K blocks kb and kb+1 are in registers; kb+2 is loaded
            // while kb is promoted, so no K block waits on a global load
            for (int kb = 0; kb < p.KB; ++kb) {
                float a2 = 0.f, g2 = 0.f, u2 = 0.f;
                if (active && kb + 2 < p.KB) {
                    a2 = __ldg(sa_row + (size_t)(kb + 2) * p.R);
                    g2 = __ldg(sw0 + kb + 2);
                    if (has1) u2 = __ldg(sw1 + kb + 2);
                }
                if (!mbar_wait(smem_u32(&tfull_bar[buf]), tphase, abort_p, err, kErrTimeoutEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the MMAs of this K block have completed, so its smem stage is free
                if (warp == 4 && lane == 0) mbar_arrive(smem_u32(&empty_bar[e_stage]));
                if (++e_stage == C::STAGES) e_stage = 0;
                if (active) {
#pragma unroll
                    for (int c = 0; c < 2 * C::HALVES; ++c) {  // 32-column pieces of each 128-column block
                        const int h = c >> 1;
                        uint32_t r[32];
                        tmem_ld32(t_lane + (uint32_t)(buf * C::BN + 128 * h + 64 * half + 32 * (c & 1)), r);
                        const float f = a0 * (h == 0 ? g0 : u0);
                        const float2 f2 = make_float2(f, f);
                        float2* a2p = reinterpret_cast<float2*>(acc + 32 * c);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            a2p[i] = __ffma2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), f2,
                                                a2p[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
                if (!ok) break;
                if (++buf == C::NBUF) {
                    buf = 0;
                    tphase ^= 1u;
                }
                a0 = a1; g0 = g1; u0 = u1;
                a1 = a2; g1 = g2; u1 = u2;
            }
            if (!ok) break;

            if (GATED) {
                // h = silu(g) * u for this thread's 64 columns of the 128-wide group
                float amax = swiglu_inplace<64>(acc, acc + 64, p.N_real - n0);
                // the row's other 64 columns belong to the partner warp (same TMEM
                // lane quarter); exchange the partial maxima through shared memory,
                // double-buffered by tile parity, behind a bounded barrier
                s_amax[tpar][half][row] = amax;
                mbar_arrive(smem_u32(&amax_bar));
                if (!mbar_wait(smem_u32(&amax_bar), tpar, abort_p, err, kErrTimeoutEpilogue)) break;
                amax = fmaxf(s_amax[tpar][0][row], s_amax[tpar][1][row]);
                const float s = group_scale(amax);
                const float rs = recip_rn(s);
                if (valid) {
                    // all 64 quotients first (independent), then the conversions and stores
                    if (quot_fast(amax)) {
                        const uint32_t keep = sign_keep(amax);
#pragma unroll
                        for (int i = 0; i < 64; ++i) acc[i] = div_fast(acc[i], s, rs, keep);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i) acc[i] = __fdiv_rn(acc[i], s);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(p.hq + (size_t)grow * p.ldq + ti.nt * 128 + 64 * half);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int i = 16 * v + 4 * q;
                            w[q] = e4m3x2(acc[i], acc[i + 1]) | (e4m3x2(acc[i + 2], acc[i + 3]) << 16);
                        }
                        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (half == 0) p.sh[(size_t)ti.nt * p.R + grow] = s;
                }
            } else {
                // w * y rows to part[slot, :].  A lane holds one row, so direct stores
                // would write 16 bytes into each of 32 rows per instruction; instead
                // each 32-row x 16-column chunk goes through shared memory and leaves
                // as 64-byte row segments, 8 rows per instruction.
                float (*stage)[20] = s_stage[GATED ? 0 : ew];
                const int sr = lane >> 2, sq = lane & 3;  // store phase: rows sr + 8i, 16-byte piece sq
                const int slot_or_skip = valid ? my_slot : -1;  // rows past the tile's rows are skipped
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    if (b == 1 && !has1) break;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float4* srow = reinterpret_cast<float4*>(&stage[lane][0]);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int i = 64 * b + 16 * c + 4 * v;
                            srow[v] = make_float4(my_w * acc[i], my_w * acc[i + 1], my_w * acc[i + 2], my_w * acc[i + 3]);
                        }
                        __syncwarp();
                        const int col = (2 * ti.nt + b) * 128 + 64 * half + 16 * c + 4 * sq;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int st = __shfl_sync(0xffffffffu, slot_or_skip, sr + 8 * i);
                            const float4 v = *reinterpret_cast<const float4*>(&stage[sr + 8 * i][4 * sq]);
                            if (st >= 0) *reinterpret_cast<float4*>(p.part + (size_t)st * p.ldp + col) = v;
                        }
                        __syncwarp();
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <bool GATED>
static cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                               cudaStream_t st) {
    using C = GemmCfg<GATED>;
    {
        // the register hand-over between warpgroups balances only at this launch count
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, moe_gemm_kernel<GATED>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    }
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_gemm_kernel<GATED>, dim3(grid), dim3(C::THREADS), (size_t)C::SMEM_BYTES, st, tmA, tmB, p);
}

cudaError_t launch_gemm_gateup(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                               cudaStream_t st) {
    return launch_gemm<true>(tmA, tmB, p, grid, st);
}

cudaError_t launch_gemm_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                             cudaStream_t st) {
    return launch_gemm<false>(tmA, tmB, p, grid, st);
}

}  // namespace moe
