// Grouped MXFP8 expert GEMMs on the block-scaled tensor-core MMA.
//
// "Hosting Qwen on Blackwell" (section "Quantization") notes that FP8 runs
// fastest on Blackwell with microscaling, one power-of-two scale for every 32
// consecutive values.  In this variant both operands carry such scales
// (UE8M0 bytes, OCP MX v1.0 section 6.3) and tcgen05.mma applies them itself
// (kind::mxf8f6f4, block_scale, scale_vec::1X):
//
//   acc[r, n] = sum_g 2^(sa[r,g]-127) * 2^(sw[n,g]-127) * sum_{k in group g} a[r,k] * w[n,k]
//
// accumulates over the whole of K in TMEM, so nothing is promoted per K
// block: the epilogue reads each tile's accumulator once.  Scale atoms
// (512 bytes = 128 rows x one 128-wide K block, mx_atom_byte layout) travel
// with their stage: global -> shared memory by bulk copy, shared memory ->
// TMEM by tcgen05.cp from the MMA thread, just before the MMAs that read them.
//
// Two tile shapes over the same tile list as the 128x128 variant:
//   prefill  128 activation rows x 256 weight rows (gate/up: the gate and the
//            up block of one 128-wide h block; down: two consecutive w2
//            blocks); A = activations, B = weights; one 256-column TMEM
//            accumulator that the epilogue drains into registers and hands
//            back before its arithmetic, so the next tile's MMAs overlap it.
//   decode   128 weight rows (gate/up: gate and up blocks) x 32 token rows;
//            A = weights, B = tokens, TMEM holds acc^T; four accumulator
//            buffers, a deep stage ring of weight bytes.
// Epilogues add the bias to the fp32 accumulator, then
//   gate/up: h = silu(g) * u, 1x32 MX requantisation -> hq codes and the
//            down GEMM's activation scale atoms;
//   down:    * routing weight -> part[t*k+j, :].
// Every mbarrier wait is bounded; a timeout sets an error bit and all roles
// drain and exit.
//
// MXFP4 weights (FP4W): "GPT-OSS on Day 0" (opening section) notes that the
// open-weight models ship with MXFP4 weights and that Blackwell's FP4 tensor
// cores run them natively.  The weight codes are E2M1, two per byte in HBM
// (half the bytes of the e4m3 codes, which is what decode-sized batches are
// bound by); the tensor map's 16U4_ALIGN16B type expands each 16-value chunk
// into the 16-byte padded form the f8f6f4 MMA kinds read, so the shared-memory
// image, the stage ring, the scale atoms and the descriptors are those of the
// e4m3 weights; what changes is the instruction descriptor's weight format and
// the byte count a weight box completes on its stage barrier (the packed
// global bytes, 8 KB per 128 x 128 box, not the 16 KB it fills).
// Activations stay MXFP8 (e4m3 codes).
#include <cuda_bf16.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// nt: the tile's (first) weight row block; two: whether a second row block,
// up_rows / 128 further on, is part of it (decode tiles)
struct MxTile {
    int e, nt, mt, row0, rows;
    bool two;
};

// Tile -> (expert, n-tile, m-tile), tiles ordered expert, n-tile, m-tile.
template <int BM>
__device__ __forceinline__ MxTile mx_tile(int tile, const int* s_tiles, const int* s_off, const int* s_cnt, int E) {
    int lo = 0, hi = E;  // s_tiles[lo] <= tile < s_tiles[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= tile)
            lo = mid;
        else
            hi = mid;
    }
    MxTile t;
    t.e = lo;
    const int local = tile - s_tiles[lo];
    const int mtc = (s_cnt[lo] + BM - 1) / BM;
    t.nt = local / mtc;
    t.mt = local - t.nt * mtc;
    t.row0 = s_off[lo] + t.mt * BM;
    t.rows = min(BM, s_cnt[lo] - t.mt * BM);
    t.two = false;
    return t;
}

// ===================================================================== prefill
template <bool GATED, bool FP4W>
struct MxCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 256;
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // bytes a stage's loads complete on its barrier: a 4-bit weight box counts its
    // packed global bytes (half its shared-memory footprint)
    static constexpr int STAGE_TX = A_BYTES + (FP4W ? B_BYTES / 2 : B_BYTES);
    static constexpr int SF_BYTES = 3 * kMxAtomBytes;  // activation tile, weight block 0, weight block 1
    static constexpr int STAGES = 4;
    static constexpr int SF_COL0 = BN;                 // TMEM: accumulator [0, 256), scale ring after it
    static constexpr int SF_STRIDE = 16;               // TMEM columns per stage (three 4-column atoms)
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARP0 = 4;  // warps 0-3: producer, MMA issuer, metadata, idle
    static constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter (warp & 3)
    static constexpr int THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
    static constexpr int SMEM_BYTES = STAGES * (STAGE_BYTES + SF_BYTES) + 1024;
    // A = activation codes (e4m3), B = weight codes (e4m3, or e2m1 for MXFP4 weights)
    static constexpr uint32_t IDESC = idesc_mx(BM, BN, kFmtE4M3, FP4W ? kFmtE2M1 : kFmtE4M3);
    static_assert(SF_COL0 + STAGES * SF_STRIDE <= TMEM_COLS, "scale ring does not fit in TMEM");
};

template <bool GATED, bool FP4W>
__global__ void __launch_bounds__(MxCfg<GATED, FP4W>::THREADS, 1)
    moe_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const MxGemmParams p) {
    using C = MxCfg<GATED, FP4W>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sf_smem = smem + C::STAGES * C::STAGE_BYTES;

    __shared__ __align__(8) uint64_t full_bar[C::STAGES];
    __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
    __shared__ __align__(8) uint64_t dfull_bar;   // accumulator complete (MMA commit)
    __shared__ __align__(8) uint64_t dempty_bar;  // accumulator drained by the epilogue warps
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ __align__(8) uint64_t bfull_bar[2];
    __shared__ __align__(8) uint64_t bempty_bar[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int s_tiles[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
    // staged one tile ahead by the metadata warp: bias, and for the down GEMM
    // each row's slot t*k+j and routing weight
    __shared__ float s_bias[2][C::BN];
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
        mbar_init(smem_u32(&dfull_bar), 1);
        mbar_init(smem_u32(&dempty_bar), C::EPI_WARPS);
        mbar_init(smem_u32(&drain_bar), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bfull_bar[b]), 32);
            mbar_init(smem_u32(&bempty_bar[b]), C::EPI_WARPS * 32);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), C::TMEM_COLS);
    pdl_wait();
    for (int i = tid; i <= E; i += C::THREADS) {
        s_tiles[i] = p.tiles[i];
        s_off[i] = p.offset[i];
        if (i < E) s_cnt[i] = p.count[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    const int total = s_tiles[E];
    volatile int* abort_p = &abort_flag;
    uint32_t* err = p.status + kStatusError;
    // no early launch_dependents at prefill sizes (see the 128x128 prefill GEMM)

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, filled = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const MxTile ti = mx_tile<C::BM>(tile, s_tiles, s_off, s_cnt, E);
                const int mtid = s_tiles[ti.e] / p.nt + ti.mt;
                const int rb0 = GATED ? ti.nt : 2 * ti.nt;
                const int rb1 = GATED ? p.up_rows / 128 + ti.nt : 2 * ti.nt + 1;
                // down GEMM with an odd block count: the last tile's second block is past the
                // expert's matrix -- its codes come from the next expert (or the tensor map's
                // zero fill), its scale atom is block 0's, and its results are dropped
                const bool has1 = rb1 < p.sw_rowblocks;
                const int blk0 = (ti.e * p.sw_rowblocks + rb0) * p.KB;
                const int blk1 = (ti.e * p.sw_rowblocks + rb1) * p.KB;
                const uint8_t* sw0 = p.sw + (size_t)blk0 * kMxAtomBytes;
                const uint8_t* sw1 = p.sw + (size_t)(has1 ? blk1 : blk0) * kMxAtomBytes;
                const uint8_t* sa = p.sa + (size_t)mtid * p.KB * kMxAtomBytes;
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, C::STAGE_TX + C::SF_BYTES);
                    const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_dst = a_dst + C::A_BYTES;
                    const uint32_t sf_dst = smem_u32(sf_smem + stage * C::SF_BYTES);
                    tma_load_2d(a_dst, &tmX, kb * 128, ti.row0, fb);
                    tma_load_2d(b_dst, &tmW, 0, (blk0 + kb) * 128, fb);
                    tma_load_2d(b_dst + 128 * 128, &tmW, 0, (blk1 + kb) * 128, fb);
                    bulk_load(sf_dst, sa + (size_t)kb * kMxAtomBytes, kMxAtomBytes, fb);
                    bulk_load(sf_dst + kMxAtomBytes, sw0 + (size_t)kb * kMxAtomBytes, kMxAtomBytes, fb);
                    bulk_load(sf_dst + 2 * kMxAtomBytes, sw1 + (size_t)kb * kMxAtomBytes, kMxAtomBytes, fb);
                    filled |= 1u << stage;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the last fill of every stage has landed, and on the normal path every
            // stage was released by an MMA commit, so nothing arrives after exit
            int dummy = 0;
            for (int i = 0; i < C::STAGES; ++i) {
                const int s = (stage + C::STAGES - 1 - i) % C::STAGES;
                const uint32_t ph = (s < stage) ? phase : phase ^ 1u;
                if (filled & (1u << s)) mbar_wait(smem_u32(&full_bar[s]), ph, &dummy, err, kErrTimeoutProducer);
            }
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
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t sphase = 0, dphase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                // the epilogue has drained the previous tile's accumulator
                if (!mbar_wait(smem_u32(&dempty_bar), dphase ^ 1u, abort_p, err, kErrTimeoutMma)) break;
                tc_fence_after();
                for (int kb = 0; kb < p.KB; ++kb) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), sphase, abort_p, err, kErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_base = a_base + C::A_BYTES;
                    const uint32_t sf_src = smem_u32(sf_smem + stage * C::SF_BYTES);
                    const uint32_t tsf = tmem_base + (uint32_t)(C::SF_COL0 + stage * C::SF_STRIDE);
                    // SFA: rows 0-127 of the tile in columns [tsf, tsf+4); SFB: weight rows
                    // 0-127 in [tsf+4, tsf+8) and 128-255 in [tsf+8, tsf+12)
                    tmem_cp_atom(tsf, sf_src);
                    tmem_cp_atom(tsf + 4, sf_src + kMxAtomBytes);
                    tmem_cp_atom(tsf + 8, sf_src + 2 * kMxAtomBytes);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_mx(tmem_base, smem_desc_sw128(a_base + 32 * k4), smem_desc_sw128(b_base + 32 * k4),
                               idesc_sf_id(C::IDESC, (uint32_t)k4), tsf, tsf + 4, (kb | k4) != 0 ? 1u : 0u);
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == C::STAGES) {
                        stage = 0;
                        sphase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&dfull_bar));
                dphase ^= 1u;
            }
            // every MMA issued above has completed before TMEM is released
            mma_commit(smem_u32(&drain_bar));
            int dummy = 0;
            mbar_wait(smem_u32(&drain_bar), 0, &dummy, err, kErrTimeoutMma);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------- metadata warp
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(smem_u32(&bempty_bar[slot]), use ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
            const MxTile t = mx_tile<C::BM>(tile, s_tiles, s_off, s_cnt, E);
            const uint16_t* bias_e = p.bias + (size_t)t.e * (GATED ? 2 * p.N_real : p.N_real);
            for (int c = lane; c < C::BN; c += 32) {
                // gate/up: h feature nt*128 + c%128 of the gate (c < 128) or up half of b13;
                // down: output feature (2nt + c/128)*128 + c%128
                const int n = (GATED ? t.nt : 2 * t.nt + (c >> 7)) * 128 + (c & 127);
                s_bias[slot][c] =
                    n < p.N_real ? bf16_bits_to_f32(__ldg(bias_e + (GATED ? (c >> 7) * p.N_real : 0) + n)) : 0.f;
            }
            if (!GATED) {
                for (int r = lane; r < 128; r += 32) {
                    const int st = __ldg(p.perm + min(t.row0 + r, p.R - 1));
                    s_rslot[slot][r] = st;
                    s_rw[slot][r] = bf16_bits_to_f32(__ldg(p.topk_wb + st));
                }
            }
            mbar_arrive(smem_u32(&bfull_bar[slot]));
        }
    } else if (warp >= C::EPI_WARP0) {
        // --------------------------------------------------------- epilogue
        const int quarter = warp & 3;                   // TMEM lanes this warp may access
        const int half = (warp - C::EPI_WARP0) >> 2;    // which 64 columns of each 128-column block
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
        uint32_t dphase = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const MxTile ti = mx_tile<C::BM>(tile, s_tiles, s_off, s_cnt, E);
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(smem_u32(&dfull_bar), dphase, abort_p, err, kErrTimeoutEpilogue)) break;
            dphase ^= 1u;
            tc_fence_after();
            float acc[128];  // block 0 (gate) columns [0, 64), block 1 (up) columns [64, 128)
            {
                uint32_t r[64];
                tmem_ld64(t_lane + (uint32_t)(64 * half), r);
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[i] = __uint_as_float(r[i]);
                tmem_ld64(t_lane + (uint32_t)(128 + 64 * half), r);
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[64 + i] = __uint_as_float(r[i]);
            }
            // the accumulator is in registers: the next tile's MMAs may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&dempty_bar));
            if (!mbar_wait(smem_u32(&bfull_bar[slot]), use, abort_p, err, kErrTimeoutEpilogue)) break;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                acc[i] += s_bias[slot][64 * half + i];
                acc[64 + i] += s_bias[slot][128 + 64 * half + i];
            }
            const int my_slot = GATED ? 0 : s_rslot[slot][GATED ? 0 : row];
            const float my_w = GATED ? 0.f : s_rw[slot][GATED ? 0 : row];
            mbar_arrive(smem_u32(&bempty_bar[slot]));
            const bool valid = row < ti.rows;
            const int grow = ti.row0 + row;

            if (GATED) {
                // h = silu(g) * u for this thread's 64 features: two 1x32 groups
                swiglu_inplace<64>(acc, acc + 64, p.N_real - (ti.nt * 128 + 64 * half));
                const int mtid = s_tiles[ti.e] / p.nt + ti.mt;
                uint32_t bytes = 0;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(acc[32 * g + i]));
                    const uint32_t sb = mx_scale_byte(amax);
                    const float inv = mx_inv_scale(sb);
                    const uint32_t keep = mx_keep(amax);
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        w[i] = mx_quant4(acc[32 * g + 4 * i], acc[32 * g + 4 * i + 1], acc[32 * g + 4 * i + 2],
                                         acc[32 * g + 4 * i + 3], inv, keep);
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(p.hq + (size_t)grow * p.ldq + ti.nt * 128 + 64 * half +
                                                              32 * g);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                    bytes |= sb << (8 * g);
                }
                // the down GEMM's activation atom of (m-tile, K block nt): groups 2*half, 2*half+1
                if (valid)
                    *reinterpret_cast<uint16_t*>(p.sh + ((size_t)mtid * (p.ldq / 128) + ti.nt) * kMxAtomBytes +
                                                 mx_atom_byte(row, 2 * half)) = (uint16_t)bytes;
            } else {
                // w * y rows to part[slot, :].  A lane holds one row, so direct stores
                // would write 16 bytes into each of 32 rows per instruction; instead
                // each 32-row x 16-column chunk goes through shared memory and leaves
                // as 64-byte row segments, 8 rows per instruction.
                const bool has1 = 2 * ti.nt + 1 < p.sw_rowblocks;
                float (*stage)[20] = s_stage[GATED ? 0 : warp - C::EPI_WARP0];
                const int sr = lane >> 2, sq = lane & 3;  // store phase: rows sr + 8i, 16-byte piece sq
                // invalid rows (past the tile's rows) get slot -1 and are skipped
                const int slot_or_skip = valid ? my_slot : -1;
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
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ====================================================================== decode
// GATED: gate and up row blocks of one n-tile per K step.  PAIRED (down GEMM
// only): w2 row blocks nt and nt + up_rows/128 per K step, as in the 128x128
// decode down GEMM; otherwise one row block, KPS K blocks per stage.
template <bool GATED, bool FP4W, bool PAIRED = false>
struct MxDecCfg {
    static constexpr bool TWO = GATED || PAIRED;  // two weight row blocks per K step
    static constexpr int BT = 32;                 // token rows per tile (MMA N)
    static constexpr int W_BYTES = (TWO ? 2 : 1) * 128 * 128;
    static constexpr int X_BYTES = BT * 128;
    // K blocks per ring stage (the ring's round trip is paid once per stage);
    // a stage holds the KPS weight blocks, then the KPS token-row blocks
    static constexpr int KPS = GATED ? MOE_MX_DEC_KPS_GATEUP : (PAIRED ? 1 : MOE_MX_DEC_KPS_DOWN);
    static constexpr int STAGE_BYTES = KPS * (W_BYTES + X_BYTES);
    static constexpr int W_TX = FP4W ? W_BYTES / 2 : W_BYTES;  // packed bytes of 4-bit weight boxes
    static constexpr int SF_KB = (TWO ? 3 : 2) * kMxAtomBytes;  // atoms of one K block: weight block(s), token tile
    static constexpr int SF_BYTES = KPS * SF_KB;
    static constexpr int MAX_STAGES = 16 / KPS;
    static constexpr int ACC_COLS = TWO ? 2 * BT : BT;
    static constexpr int NACC = 4;  // accumulator buffers
    static constexpr int SF_COL0 = 256;
    static constexpr int SF_STRIDE = 16 * KPS;  // TMEM scale columns of one stage (16 per K block)
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_WARPS = 4;
    static constexpr int META_WARP = 6;
    static constexpr int THREADS = 7 * 32;
    // A = weight codes (e4m3, or e2m1 for MXFP4 weights), B = token codes (e4m3)
    static constexpr uint32_t IDESC = idesc_mx(128, BT, FP4W ? kFmtE2M1 : kFmtE4M3, kFmtE4M3);
    static_assert(NACC * ACC_COLS <= SF_COL0, "accumulators overlap the scale ring");
    static_assert(SF_COL0 + MAX_STAGES * SF_STRIDE <= TMEM_COLS, "scale ring does not fit in TMEM");
};

// Decode tile -> (expert, row block(s), m-tile): the order of mx_tile, except
// for paired down tiles (P = up_rows / 128 > 0), where of the nt = RB - P
// n-tiles of an m-tile the first P take w2 row blocks j and j + P and the
// other RB - 2P one block each, every m-tile's paired tiles listed before all
// the one-block ones (the layout of the 128x128 decode down GEMM's list).
template <bool GATED, bool PAIRED, int BM>
__device__ __forceinline__ MxTile mx_dec_tile(int tile, const int* s_tiles, const int* s_off, const int* s_cnt, int E,
                                              const MxGemmParams& p) {
    if (!PAIRED) {
        MxTile t = mx_tile<BM>(tile, s_tiles, s_off, s_cnt, E);
        t.two = GATED;
        return t;
    }
    const int P = p.up_rows / 128, NT = p.nt, S = NT - P;
    const int mtt = s_tiles[E] / NT;  // m-tiles of all experts
    int g, nt;
    if (tile < P * mtt) {
        g = tile / P;
        nt = tile - g * P;
    } else {
        const int r = tile - P * mtt;  // S > 0 here
        g = r / S;
        nt = P + (r - g * S);
    }
    int lo = 0, hi = E;  // s_tiles[lo] / NT <= g < s_tiles[hi] / NT
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= g * NT)
            lo = mid;
        else
            hi = mid;
    }
    MxTile t;
    t.e = lo;
    t.mt = g - s_tiles[lo] / NT;
    t.nt = nt < P ? nt : nt + P;
    t.two = nt < P;
    t.row0 = s_off[lo] + t.mt * BM;
    t.rows = min(BM, s_cnt[lo] - t.mt * BM);
    return t;
}

template <bool GATED, bool FP4W, bool PAIRED>
__global__ void __launch_bounds__(MxDecCfg<GATED, FP4W, PAIRED>::THREADS, 1)
    moe_gemm_mx_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                              const MxGemmParams p, const int nst) {
    using C = MxDecCfg<GATED, FP4W, PAIRED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* sf_smem = smem + nst * C::STAGE_BYTES;

    __shared__ __align__(8) uint64_t full_bar[C::MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[C::MAX_STAGES];
    __shared__ __align__(8) uint64_t dfull_bar[C::NACC];
    __shared__ __align__(8) uint64_t dempty_bar[C::NACC];
    __shared__ __align__(8) uint64_t mfull_bar[2];
    __shared__ __align__(8) uint64_t mempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int s_tiles[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
    __shared__ float s_bias[2][C::TWO ? 256 : 128];
    __shared__ int s_slot[2][32];
    __shared__ float s_w[2][32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < C::NACC; ++b) {
            mbar_init(smem_u32(&dfull_bar[b]), 1);
            mbar_init(smem_u32(&dempty_bar[b]), C::EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&mfull_bar[b]), 32);
            mbar_init(smem_u32(&mempty_bar[b]), C::EPI_WARPS * 32);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), C::TMEM_COLS);
    pdl_wait();
    for (int i = tid; i <= E; i += C::THREADS) {
        s_tiles[i] = p.tiles[i];
        s_off[i] = p.offset[i];
        if (i < E) s_cnt[i] = p.count[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    const int total = s_tiles[E];
    volatile int* abort_p = &abort_flag;
    uint32_t* err = p.status + kStatusError;
    pdl_allow_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, filled = 0;
            bool ok = true;
            const int ublk = (p.up_rows / 128) * p.KB;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const MxTile ti = mx_dec_tile<GATED, PAIRED, C::BT>(tile, s_tiles, s_off, s_cnt, E, p);
                const int mtid = s_tiles[ti.e] / p.nt + ti.mt;
                const int wblk = (ti.e * p.sw_rowblocks + ti.nt) * p.KB;
                const bool two = C::TWO && ti.two;
                const int nxb = (ti.rows + kDecXBoxRows - 1) / kDecXBoxRows;
                const uint8_t* sa = p.sa + (size_t)mtid * p.KB * kMxAtomBytes;
                for (int kb0 = 0; kb0 < p.KB; kb0 += C::KPS) {
                    const int nk = min(C::KPS, p.KB - kb0);
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    // one weight box and one scale atom fewer when a paired tile has no second block
                    const int miss = C::TWO && !two ? C::W_TX / 2 + kMxAtomBytes : 0;
                    mbar_arrive_expect_tx(fb, nk * (C::W_TX + nxb * kDecXBoxRows * 128 + C::SF_KB - miss));
                    for (int i = 0; i < nk; ++i) {
                        const int kb = kb0 + i;
                        const uint32_t w_dst = smem_u32(smem + stage * C::STAGE_BYTES + i * C::W_BYTES);
                        const uint32_t x_dst = smem_u32(smem + stage * C::STAGE_BYTES + C::KPS * C::W_BYTES +
                                                        i * C::X_BYTES);
                        const uint32_t sf_dst = smem_u32(sf_smem + stage * C::SF_BYTES + i * C::SF_KB);
                        tma_load_2d(w_dst, &tmW, 0, (wblk + kb) * 128, fb);
                        bulk_load(sf_dst, p.sw + (size_t)(wblk + kb) * kMxAtomBytes, kMxAtomBytes, fb);
                        if (two) {
                            tma_load_2d(w_dst + 128 * 128, &tmW, 0, (wblk + ublk + kb) * 128, fb);
                            bulk_load(sf_dst + kMxAtomBytes, p.sw + (size_t)(wblk + ublk + kb) * kMxAtomBytes,
                                      kMxAtomBytes, fb);
                        }
                        // only the boxes that hold rows of this tile; the MMA reads stale shared
                        // memory for the other token columns, whose results are never stored
                        for (int b = 0; b < nxb; ++b)
                            tma_load_2d(x_dst + b * kDecXBoxRows * 128, &tmX, kb * 128, ti.row0 + b * kDecXBoxRows, fb);
                        bulk_load(sf_dst + (C::TWO ? 2 : 1) * kMxAtomBytes, sa + (size_t)kb * kMxAtomBytes,
                                  kMxAtomBytes, fb);
                    }
                    filled |= 1u << stage;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            int dummy = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = (stage + nst - 1 - i) % nst;
                const uint32_t ph = (s < stage) ? phase : phase ^ 1u;
                if (filled & (1u << s)) mbar_wait(smem_u32(&full_bar[s]), ph, &dummy, err, kErrTimeoutProducer);
            }
            if (ok) {
                for (int i = 0; i < nst; ++i) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
                    if (++stage == nst) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            int stage = 0, buf = 0;
            uint32_t sphase = 0, aphase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const bool two = C::TWO && mx_dec_tile<GATED, PAIRED, C::BT>(tile, s_tiles, s_off, s_cnt, E, p).two;
                if (!mbar_wait(smem_u32(&dempty_bar[buf]), aphase ^ 1u, abort_p, err, kErrTimeoutMma)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * C::ACC_COLS);
                for (int kb0 = 0; kb0 < p.KB; kb0 += C::KPS) {
                    const int nk = min(C::KPS, p.KB - kb0);
                    if (!mbar_wait(smem_u32(&full_bar[stage]), sphase, abort_p, err, kErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int i = 0; i < nk; ++i) {
                        const int kb = kb0 + i;
                        const uint32_t w_base = smem_u32(smem + stage * C::STAGE_BYTES + i * C::W_BYTES);
                        const uint32_t x_base = smem_u32(smem + stage * C::STAGE_BYTES + C::KPS * C::W_BYTES +
                                                         i * C::X_BYTES);
                        const uint32_t sf_src = smem_u32(sf_smem + stage * C::SF_BYTES + i * C::SF_KB);
                        const uint32_t tsf = tmem_base + (uint32_t)(C::SF_COL0 + stage * C::SF_STRIDE + 16 * i);
                        // SFA: gate (or only) block [tsf, tsf+4), up block [tsf+4, tsf+8); SFB: tokens [tsf+8, ...)
                        tmem_cp_atom(tsf, sf_src);
                        if (two) tmem_cp_atom(tsf + 4, sf_src + kMxAtomBytes);
                        tmem_cp_atom(tsf + 8, sf_src + (C::TWO ? 2 : 1) * kMxAtomBytes);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint64_t xd = smem_desc_sw128(x_base + 32 * k4);
                            const uint32_t id = idesc_sf_id(C::IDESC, (uint32_t)k4);
                            const uint32_t acc = (kb | k4) != 0 ? 1u : 0u;
                            mma_mx(d, smem_desc_sw128(w_base + 32 * k4), xd, id, tsf, tsf + 8, acc);
                            if (two)
                                mma_mx(d + C::BT, smem_desc_sw128(w_base + 128 * 128 + 32 * k4), xd, id, tsf + 4,
                                       tsf + 8, acc);
                        }
                    }
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == nst) {
                        stage = 0;
                        sphase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&dfull_bar[buf]));
                if (++buf == C::NACC) {
                    buf = 0;
                    aphase ^= 1u;
                }
            }
            mma_commit(smem_u32(&drain_bar));
            int dummy = 0;
            mbar_wait(smem_u32(&drain_bar), 0, &dummy, err, kErrTimeoutMma);
        }
    } else if (warp == C::META_WARP) {
        // --------------------------------------------------- metadata warp
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(smem_u32(&mempty_bar[slot]), use ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
            const MxTile ti = mx_dec_tile<GATED, PAIRED, C::BT>(tile, s_tiles, s_off, s_cnt, E, p);
            const uint16_t* bias_e = p.bias + (size_t)ti.e * (GATED ? 2 * p.N_real : p.N_real);
            // bias of the tile's features: [0, 128) first row block, [128, 256) second
#pragma unroll
            for (int c = lane; c < (C::TWO ? 256 : 128); c += 32) {
                const int n = ti.nt * 128 + (c & 127) + (GATED ? 0 : (c >> 7) * p.up_rows);
                s_bias[slot][c] =
                    n < p.N_real ? bf16_bits_to_f32(__ldg(bias_e + (GATED ? (c >> 7) * p.N_real : 0) + n)) : 0.f;
            }
            if (!GATED) {
                const int st = __ldg(p.perm + min(ti.row0 + lane, p.R - 1));
                s_slot[slot][lane] = st;
                s_w[slot][lane] = bf16_bits_to_f32(__ldg(p.topk_wb + st));
            }
            mbar_arrive(smem_u32(&mfull_bar[slot]));
        }
    } else if (warp >= 2 && warp < 2 + C::EPI_WARPS) {
        // --------------------------------------------------------- epilogue
        const int quarter = warp & 3;        // TMEM lanes this warp may access
        const int nl = quarter * 32 + lane;  // output feature within the 128-wide n-tile
        const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int buf = 0, it = 0;
        uint32_t aphase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(smem_u32(&dfull_bar[buf]), aphase, abort_p, err, kErrTimeoutEpilogue)) break;
            tc_fence_after();
            float acc[C::ACC_COLS];  // column j: token j (gate/up: gate [0, 32), up [32, 64); paired likewise)
            {
                const uint32_t tcol = t_lane + (uint32_t)(buf * C::ACC_COLS);
                if (C::TWO) {
                    uint32_t r[64];
                    tmem_ld64(tcol, r);
#pragma unroll
                    for (int j = 0; j < C::ACC_COLS; ++j) acc[j] = __uint_as_float(r[j]);
                } else {
                    uint32_t r[32];
                    tmem_ld32(tcol, r);
#pragma unroll
                    for (int j = 0; j < C::ACC_COLS; ++j) acc[j] = __uint_as_float(r[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[buf]));
            if (++buf == C::NACC) {
                buf = 0;
                aphase ^= 1u;
            }
            if (!mbar_wait(smem_u32(&mfull_bar[slot]), use, abort_p, err, kErrTimeoutEpilogue)) break;
            const MxTile ti = mx_dec_tile<GATED, PAIRED, C::BT>(tile, s_tiles, s_off, s_cnt, E, p);
            const int n = ti.nt * 128 + nl;
            {
                const float bg = s_bias[slot][nl];
                const float bu = C::TWO ? s_bias[slot][C::TWO ? 128 + nl : 0] : 0.f;
#pragma unroll
                for (int j = 0; j < C::BT; ++j) {
                    acc[j] += bg;
                    if (C::TWO) acc[C::BT + j] += bu;
                }
            }
            if (GATED) {
                mbar_arrive(smem_u32(&mempty_bar[slot]));
                swiglu_inplace<32>(acc, acc + 32, n < p.N_real ? 32 : 0);
                // the 1x32 group of token j is this warp's 32 features: its amax is column j's max
                float habs[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) habs[j] = fabsf(acc[j]);
                const float amax = column_max32(habs, lane);  // lane j: token j
                const uint32_t sb = mx_scale_byte(amax);
                const float inv = mx_inv_scale(sb);
                const uint32_t keep = mx_keep(amax);
                if (lane < ti.rows) {
                    const int mtid = s_tiles[ti.e] / p.nt + ti.mt;
                    p.sh[((size_t)mtid * (p.ldq / 128) + ti.nt) * kMxAtomBytes + mx_atom_byte(lane, quarter)] =
                        (uint8_t)sb;
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const uint32_t codes =
                        e4m3x2(mx_scaled(acc[j], __shfl_sync(0xffffffffu, inv, j), __shfl_sync(0xffffffffu, keep, j)),
                               mx_scaled(acc[j + 1], __shfl_sync(0xffffffffu, inv, j + 1),
                                         __shfl_sync(0xffffffffu, keep, j + 1)));
                    if (j < ti.rows) p.hq[(size_t)(ti.row0 + j) * p.ldq + n] = (uint8_t)(codes & 0xffu);
                    if (j + 1 < ti.rows) p.hq[(size_t)(ti.row0 + j + 1) * p.ldq + n] = (uint8_t)(codes >> 8);
                }
            } else {
                const int slot_l = s_slot[slot][lane];
                const float w_l = s_w[slot][lane];
                mbar_arrive(smem_u32(&mempty_bar[slot]));
                const bool two = C::TWO && ti.two;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int slot_t = __shfl_sync(0xffffffffu, slot_l, j);
                    const float w = __shfl_sync(0xffffffffu, w_l, j);
                    if (j < ti.rows) {
                        p.part[(size_t)slot_t * p.ldp + n] = w * acc[j];
                        if (two) p.part[(size_t)slot_t * p.ldp + n + p.up_rows] = w * acc[C::BT + j];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ===================================================================== launch
template <bool GATED, bool FP4W>
static cudaError_t launch_mx_prefill(const CUtensorMap& tmX, const CUtensorMap& tmW, const MxGemmParams& p, int grid,
                                     cudaStream_t st) {
    using C = MxCfg<GATED, FP4W>;
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_mx_kernel<GATED, FP4W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_gemm_mx_kernel<GATED, FP4W>, dim3(grid), dim3(C::THREADS), (size_t)C::SMEM_BYTES, st, tmX,
                      tmW, p);
}

// The stage ring takes the shared memory the kernel's static arrays leave, up
// to `max_stages` stages.
template <bool GATED, bool FP4W, bool PAIRED>
static cudaError_t launch_mx_decode(const CUtensorMap& tmX, const CUtensorMap& tmW, const MxGemmParams& p, int grid,
                                    int max_stages, cudaStream_t st) {
    using C = MxDecCfg<GATED, FP4W, PAIRED>;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, moe_gemm_mx_decode_kernel<GATED, FP4W, PAIRED>);
    if (e != cudaSuccess) return e;
    const long long room = (long long)optin - (long long)fa.sharedSizeBytes - 1024;
    int nst = (int)(room / (C::STAGE_BYTES + C::SF_BYTES));
    if (nst > max_stages) nst = max_stages;
    if (nst > C::MAX_STAGES) nst = C::MAX_STAGES;
    if (nst < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)nst * (C::STAGE_BYTES + C::SF_BYTES) + 1024;
    e = cudaFuncSetAttribute(moe_gemm_mx_decode_kernel<GATED, FP4W, PAIRED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_gemm_mx_decode_kernel<GATED, FP4W, PAIRED>, dim3(grid), dim3(C::THREADS), smem, st, tmX, tmW, p,
                      nst);
}

template <bool FP4W>
static cudaError_t launch_mx(bool gated, bool decode, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             const MxGemmParams& p, int grid, cudaStream_t st) {
    if (decode)
        return gated            ? launch_mx_decode<true, FP4W, false>(tmX, tmW, p, grid, kDecStagesGateUp, st)
               : p.up_rows != 0 ? launch_mx_decode<false, FP4W, true>(tmX, tmW, p, grid, kDecStagesGateUp, st)
                                : launch_mx_decode<false, FP4W, false>(tmX, tmW, p, grid, kDecStagesDown, st);
    return gated ? launch_mx_prefill<true, FP4W>(tmX, tmW, p, grid, st)
                 : launch_mx_prefill<false, FP4W>(tmX, tmW, p, grid, st);
}

cudaError_t launch_gemm_mx(bool gated, bool decode, bool fp4w, const CUtensorMap& tmX, const CUtensorMap& tmW,
                           const MxGemmParams& p, int grid, cudaStream_t st) {
    return fp4w ? launch_mx<true>(gated, decode, tmX, tmW, p, grid, st)
                : launch_mx<false>(gated, decode, tmX, tmW, p, grid, st);
}

}  // namespace moe
