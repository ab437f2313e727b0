// Grouped FP8 expert GEMMs for decode-sized batches (few rows per expert).
//
// Same arithmetic as the prefill kernels (moe_gemm.cu):
//   acc[r, n] = bias[n] + sum_kb (sa[kb, r] * sw[n/128, kb]) * P_kb[r, n]
// but with the operands swapped: the expert's weight rows are the MMA's M=128
// operand and at most 32 token rows of that expert are the N=32 operand, so
// TMEM holds acc^T (lane = output feature, column = token).  Decode is bound
// by streaming the activated experts' weights from HBM ("Hosting Qwen on
// Blackwell", Decoders: with few tokens the GEMM is limited by loading
// weights into the tensor cores), so nearly all of every pipeline stage is
// weight bytes: 5 stages of two 16 KB weight blocks are in flight per SM --
// deeper rings were measured and gain nothing -- and the small TMEM tiles
// give 8-16 accumulation buffers, so the scale promotion never stalls the
// MMA.  A tile loads only the 8-row boxes of token rows it has; the metadata
// slots are sized by the K-block count.
//
// Tile = (expert, 128 output features -- 256 for the gate/up GEMM's gate and
// up halves and for the paired down GEMM -- and 32 token rows), ordered
// expert, n-tile, m-tile; one CTA per SM, persistent.  Two weight blocks per
// K step stream faster than one: with one 16 KB block per stage the down
// GEMM's stages arrived every ~0.48 us whatever the ring depth (9 or 5
// stages), with two every ~0.75 us.  So the down GEMM pairs w2 row blocks j
// and j + P in its first P n-tiles, P chosen at launch for the balance of
// the tile list over the SMs (0 -- one block per tile -- when one-block
// tiles would not even fill them).
//
//   warp 0     TMA producer (weights: one or two 128x128 boxes; tokens: the
//              tile's rows in boxes of 8)
//   warp 1     TMEM allocator and MMA issuer
//   warps 2-5  promotion + epilogue, one TMEM lane quarter (32 features) each:
//              gate/up: h = silu(g)*u, 1x128 requant across the 128 features of
//              a token (column max by shuffles + shared memory), codes -> hq,
//              scales -> sh;  down: * routing weight -> part[t*k+j, n]
//   warp 6     metadata: stages each tile's bias, token scales, weight scales
//              (and, for the down GEMM, the tokens' slots and routing weights)
//              in shared memory one tile ahead, so neither the promotion nor
//              the epilogue waits on global memory and a tile's epilogue is
//              short enough for the MMA to run on into the next tile.
#include <cuda_bf16.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// GATED: the gate/up GEMM (gate and up row blocks of one n-tile per K step).
// PAIRED (down GEMM only): two w2 row blocks per K step, nt and nt + U with
// U = ceil(row blocks / 2), 256 output features per tile.
template <bool GATED, bool PAIRED = false>
struct DecCfg {
    static constexpr bool TWO = GATED || PAIRED;          // two weight row blocks per K step
    static constexpr int BT = 32;                         // token rows per tile (MMA N)
    static constexpr int W_BYTES = (TWO ? 2 : 1) * 128 * 128;
    static constexpr int X_BYTES = BT * 128;
    // K blocks per ring stage (one: two per stage were measured slower for both
    // GEMMs, which stream at their bound with one)
    static constexpr int KPS = GATED ? MOE_DEC_KPS_GATEUP : MOE_DEC_KPS_DOWN;
    // stage: the KPS weight blocks, then the KPS token-row blocks
    static constexpr int STAGE_BYTES = KPS * (W_BYTES + X_BYTES);
    static constexpr int MAX_STAGES = 16;                 // the ring takes what shared memory is left (launch)
    static constexpr int ACC_COLS = TWO ? 2 * BT : BT;    // TMEM columns of one accumulation buffer
    static constexpr int TMEM_COLS = 512;
    static constexpr int NBUF = TMEM_COLS / ACC_COLS;     // 8 (two row blocks) or 16
    static constexpr int EPI_WARPS = 4;
    static constexpr int META_WARP = 6;
    static constexpr int THREADS = 7 * 32;
    static constexpr uint32_t IDESC = idesc_e4m3_f32(128, BT);
};

// nt: the tile's (first) weight row block within the expert; two: whether a
// second row block, up_rows / 128 further on, is part of it
struct DecTile {
    int e, nt, row0, rows;
    bool two;
};

// One metadata slot (floats), sized by the K-block count: bias [256], token
// scales [KB][32], weight scales of the gate (or only) block [KB] and of the
// up block [KB], token slots [32] (int) and routing weights [32].
struct DecMeta {
    int sa, sw, swu, slot, w, floats;
};
__host__ __device__ inline DecMeta dec_meta(int KB) {
    DecMeta m;
    m.sa = 256;
    m.sw = m.sa + 32 * KB;
    m.swu = m.sw + KB;
    m.slot = m.swu + KB;
    m.w = m.slot + 32;
    m.floats = (m.w + 32 + 3) & ~3;
    return m;
}

__device__ __forceinline__ DecTile decode_dec_tile(int tile, const int* s_tiles, const int* s_off, const int* s_cnt,
                                                   int E) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= tile)
            lo = mid;
        else
            hi = mid;
    }
    DecTile ti;
    ti.e = lo;
    const int local = tile - s_tiles[lo];
    const int mtc = (s_cnt[lo] + 31) >> 5;
    ti.nt = local / mtc;
    const int mt = local - ti.nt * mtc;
    ti.row0 = s_off[lo] + mt * 32;
    ti.rows = min(32, s_cnt[lo] - mt * 32);
    return ti;
}

// Tile -> (expert, row block(s), m-tile).  Gate/up and one-block down tiles:
// the list is ordered expert, n-tile, m-tile (decode_dec_tile).  Paired down
// tiles (P = up_rows / 128 > 0): of the NT = RB - P n-tiles of an m-tile, the
// first P take w2 row blocks j and j + P, the other RB - 2P one block each
// (2P .. RB-1); the list holds every m-tile's P paired tiles (m-tile by
// m-tile, expert order) before all the one-block ones, so that a round-robin
// assignment gives no CTA more paired tiles than another has plus one.
// Weight block (e, row block, kb) starts at row ((e*RB + rb)*KB + kb)*128.
template <bool GATED, bool PAIRED>
__device__ __forceinline__ DecTile dec_tile(int tile, const int* s_tiles, const int* s_off, const int* s_cnt, int E,
                                            const GemmParams& p) {
    if (!PAIRED) {
        DecTile t = decode_dec_tile(tile, s_tiles, s_off, s_cnt, E);
        t.two = GATED;
        return t;
    }
    const int P = p.up_rows / 128, NT = p.sw_rowblocks - P, S = NT - P;
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
    const int mt = g - s_tiles[lo] / NT;
    DecTile t;
    t.e = lo;
    t.nt = nt < P ? nt : nt + P;
    t.two = nt < P;
    t.row0 = s_off[lo] + mt * 32;
    t.rows = min(32, s_cnt[lo] - mt * 32);
    return t;
}

template <bool GATED, bool PAIRED>
__global__ void __launch_bounds__(DecCfg<GATED, PAIRED>::THREADS, 1)
    moe_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                           const GemmParams p, const int nst) {
    using C = DecCfg<GATED, PAIRED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const DecMeta M = dec_meta(p.KB);
    float* meta = reinterpret_cast<float*>(smem + nst * C::STAGE_BYTES);  // [2][M.floats]

    __shared__ __align__(8) uint64_t full_bar[C::MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[C::MAX_STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[C::NBUF];
    __shared__ __align__(8) uint64_t tempty_bar[C::NBUF];
    __shared__ __align__(8) uint64_t mfull_bar[2];
    __shared__ __align__(8) uint64_t mempty_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ __align__(8) uint64_t amax_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int s_tiles[kMaxExperts + 1], s_off[kMaxExperts + 1], s_cnt[kMaxExperts];
    __shared__ float s_amax[2][4][32];  // [tile parity][lane quarter][token]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(smem_u32(&tfull_bar[b]), 1);
            mbar_init(smem_u32(&tempty_bar[b]), C::EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&mfull_bar[b]), 32);
            mbar_init(smem_u32(&mempty_bar[b]), C::EPI_WARPS * 32);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        mbar_init(smem_u32(&amax_bar), C::EPI_WARPS * 32);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), C::TMEM_COLS);
    // The tile lists come from the router's scan, which had completed before
    // the kernel ahead of this one let it be scheduled; read them from L2 now.
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
    // output (the token rows) it loads after the wait.
    int pre = 0;  // stages whose weight boxes are in flight before the wait
    if (warp == 0 && lane == 0) {
        for (int tile = blockIdx.x; tile < total && pre < nst; tile += gridDim.x) {
            const DecTile ti = dec_tile<GATED, PAIRED>(tile, s_tiles, s_off, s_cnt, E, p);
            const int wblk = (ti.e * p.sw_rowblocks + ti.nt) * p.KB;
            const int ublk = (p.up_rows / 128) * p.KB;
            const bool two = ti.two;
            const int nxb = (ti.rows + kDecXBoxRows - 1) / kDecXBoxRows;
            for (int kb = 0; kb < p.KB && pre < nst; kb += C::KPS, ++pre) {
                const int nk = min(C::KPS, p.KB - kb);
                const uint32_t fb = smem_u32(&full_bar[pre]);
                mbar_arrive_expect_tx(fb, nk * ((two ? 2 : 1) * 128 * 128 + nxb * kDecXBoxRows * 128));
                for (int i = 0; i < nk; ++i) {
                    const uint32_t w_dst = smem_u32(smem + pre * C::STAGE_BYTES + i * C::W_BYTES);
                    tma_load_2d(w_dst, &tmW, 0, (wblk + kb + i) * 128, fb);
                    if (C::TWO && two) tma_load_2d(w_dst + 128 * 128, &tmW, 0, (wblk + ublk + kb + i) * 128, fb);
                }
            }
        }
    }
    pdl_wait();
    pdl_allow_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, filled = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const DecTile ti = dec_tile<GATED, PAIRED>(tile, s_tiles, s_off, s_cnt, E, p);
                const int wblk = (ti.e * p.sw_rowblocks + ti.nt) * p.KB;
                const int ublk = (p.up_rows / 128) * p.KB;
                const bool two = ti.two;
                const int nxb = (ti.rows + kDecXBoxRows - 1) / kDecXBoxRows;
                for (int kb = 0; kb < p.KB; kb += C::KPS) {
                    const int nk = min(C::KPS, p.KB - kb);
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    const uint32_t s_base = smem_u32(smem + stage * C::STAGE_BYTES);
                    if (pre > 0) {
                        --pre;  // first use of this stage: its weights went out before the wait
                    } else {
                        if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(fb, nk * ((two ? 2 : 1) * 128 * 128 + nxb * kDecXBoxRows * 128));
                        for (int i = 0; i < nk; ++i) {
                            const uint32_t w_dst = s_base + i * C::W_BYTES;
                            tma_load_2d(w_dst, &tmW, 0, (wblk + kb + i) * 128, fb);
                            if (C::TWO && two)
                                tma_load_2d(w_dst + 128 * 128, &tmW, 0, (wblk + ublk + kb + i) * 128, fb);
                        }
                    }
                    // only the boxes that hold rows of this tile; the MMA reads stale shared
                    // memory for the other token columns, whose results are never stored
                    for (int i = 0; i < nk; ++i)
                        for (int b = 0; b < nxb; ++b)
                            tma_load_2d(s_base + C::KPS * C::W_BYTES + i * C::X_BYTES + b * kDecXBoxRows * 128, &tmX,
                                        (kb + i) * 128, ti.row0 + b * kDecXBoxRows, fb);
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
            uint32_t sphase = 0, tphase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const bool two = C::TWO && dec_tile<GATED, PAIRED>(tile, s_tiles, s_off, s_cnt, E, p).two;
                for (int kb = 0; kb < p.KB && ok; kb += C::KPS) {
                    const int nk = min(C::KPS, p.KB - kb);
                    if (!mbar_wait(smem_u32(&full_bar[stage]), sphase, abort_p, err, kErrTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    const uint32_t s_base = smem_u32(smem + stage * C::STAGE_BYTES);
                    // each K block of the stage into its own TMEM buffer (promoted separately)
                    for (int i = 0; i < nk; ++i) {
                        if (!mbar_wait(smem_u32(&tempty_bar[buf]), tphase ^ 1u, abort_p, err, kErrTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t w_base = s_base + i * C::W_BYTES;
                        const uint32_t x_base = s_base + C::KPS * C::W_BYTES + i * C::X_BYTES;
                        const uint32_t d = tmem_base + (uint32_t)(buf * C::ACC_COLS);
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint64_t xd = smem_desc_sw128(x_base + 32 * k4);
                            mma_e4m3(d, smem_desc_sw128(w_base + 32 * k4), xd, C::IDESC, k4 > 0 ? 1u : 0u);
                            if (two)
                                mma_e4m3(d + C::BT, smem_desc_sw128(w_base + 128 * 128 + 32 * k4), xd, C::IDESC,
                                         k4 > 0 ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&tfull_bar[buf]));
                        if (++buf == C::NBUF) {
                            buf = 0;
                            tphase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == nst) {
                        stage = 0;
                        sphase ^= 1u;
                    }
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
            const uint32_t use = (uint32_t)(it >> 1) & 1u;  // parity of this slot's use
            if (!mbar_wait(smem_u32(&mempty_bar[slot]), use ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
            float* m = meta + slot * M.floats;
            const DecTile ti = dec_tile<GATED, PAIRED>(tile, s_tiles, s_off, s_cnt, E, p);
            const bool two = ti.two;
            const uint16_t* bias_e = p.bias + (size_t)ti.e * (GATED ? 2 * p.N_real : p.N_real);
            // bias of the tile's features: [0, 128) first row block, [128, 256) second
#pragma unroll
            for (int c = lane; c < (C::TWO ? 256 : 128); c += 32) {
                const int n = ti.nt * 128 + (c & 127) + (GATED ? 0 : (c >> 7) * p.up_rows);
                m[c] = n < p.N_real ? bf16_bits_to_f32(__ldg(bias_e + (GATED ? (c >> 7) * p.N_real : 0) + n)) : 0.f;
            }
            const int rtok = min(ti.row0 + lane, p.R - 1);
            // the tile's token scales, eight K blocks in flight per lane
            for (int kb = 0; kb < p.KB; kb += 8) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = kb + i < p.KB ? __ldg(p.sa + (size_t)(kb + i) * p.R + rtok) : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (kb + i < p.KB) m[M.sa + (kb + i) * 32 + lane] = v[i];
            }
            const float* sw_g = p.sw + ((size_t)ti.e * p.sw_rowblocks + ti.nt) * p.KB;
            for (int kb = lane; kb < p.KB; kb += 32) {
                m[M.sw + kb] = __ldg(sw_g + kb);
                if (C::TWO) m[M.swu + kb] = two ? __ldg(sw_g + (p.up_rows / 128) * p.KB + kb) : 0.f;
            }
            if (!GATED) {
                const int slot_t = __ldg(p.perm + rtok);
                reinterpret_cast<int*>(m)[M.slot + lane] = slot_t;
                m[M.w + lane] = bf16_bits_to_f32(__ldg(p.topk_wb + slot_t));
            }
            mbar_arrive(smem_u32(&mfull_bar[slot]));
        }
    } else if (warp >= 2 && warp < 2 + C::EPI_WARPS) {
        // -------------------------------------------- promotion + epilogue
        const int quarter = warp & 3;            // TMEM lanes this warp may access
        const int nl = quarter * 32 + lane;      // output feature within the 128-wide n-tile
        const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
        int buf = 0, it = 0;
        uint32_t tphase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
            const int slot = it & 1;
            const uint32_t use = (uint32_t)(it >> 1) & 1u;
            const uint32_t tpar = (uint32_t)it & 1u;
            if (!mbar_wait(smem_u32(&mfull_bar[slot]), use, abort_p, err, kErrTimeoutEpilogue)) break;
            const float* m = meta + slot * M.floats;
            const DecTile ti = dec_tile<GATED, PAIRED>(tile, s_tiles, s_off, s_cnt, E, p);
            const int n = ti.nt * 128 + nl;
            const bool nvalid = n < p.N_real;
            float acc[C::ACC_COLS];
            {
                const float bg = m[nl];
                const float bu = C::TWO ? m[128 + nl] : 0.f;
#pragma unroll
                for (int j = 0; j < C::BT; ++j) {
                    acc[j] = bg;
                    if (C::TWO) acc[C::BT + j] = bu;
                }
            }
            for (int kb = 0; kb < p.KB; ++kb) {
                if (!mbar_wait(smem_u32(&tfull_bar[buf]), tphase, abort_p, err, kErrTimeoutEpilogue)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tcol = t_lane + (uint32_t)(buf * C::ACC_COLS);
                const float a = m[M.sa + kb * 32 + lane];  // lane j: scale of token j in this K block
                const float fg = a * m[M.sw + kb];
                if (C::TWO) {
                    const float fu = a * m[M.swu + kb];
                    uint32_t r[64];
                    tmem_ld64(tcol, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float sg = __shfl_sync(0xffffffffu, fg, j);
                        const float su = __shfl_sync(0xffffffffu, fu, j);
                        acc[j] = fmaf(__uint_as_float(r[j]), sg, acc[j]);
                        acc[32 + j] = fmaf(__uint_as_float(r[32 + j]), su, acc[32 + j]);
                    }
                } else {
                    uint32_t r[32];
                    tmem_ld32(tcol, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float sg = __shfl_sync(0xffffffffu, fg, j);
                        acc[j] = fmaf(__uint_as_float(r[j]), sg, acc[j]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[buf]));
                if (++buf == C::NBUF) {
                    buf = 0;
                    tphase ^= 1u;
                }
            }
            if (!ok) break;

            if (GATED) {
                mbar_arrive(smem_u32(&mempty_bar[slot]));  // this tile's metadata is no longer read
                // h = silu(g) * u; per-token amax over the 128 features (4 warps x 32 lanes)
                swiglu_inplace<32>(acc, acc + 32, nvalid ? 32 : 0);
                float habs[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) habs[j] = fabsf(acc[j]);
                s_amax[tpar][quarter][lane] = column_max32(habs, lane);  // lane j: this warp's max for token j
                mbar_arrive(smem_u32(&amax_bar));
                if (!mbar_wait(smem_u32(&amax_bar), tpar, abort_p, err, kErrTimeoutEpilogue)) break;
                const float amax = fmaxf(fmaxf(s_amax[tpar][0][lane], s_amax[tpar][1][lane]),
                                         fmaxf(s_amax[tpar][2][lane], s_amax[tpar][3][lane]));
                const float s_tok = group_scale(amax);  // lane j: scale of token j
                const float r_tok = recip_rn(s_tok);
                if (quarter == 0 && lane < ti.rows) p.sh[(size_t)ti.nt * p.R + ti.row0 + lane] = s_tok;
                if (__all_sync(0xffffffffu, quot_fast(amax) || lane >= ti.rows)) {  // token columns past the tile's rows are never stored
                    const uint32_t k_tok = sign_keep(amax);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        acc[j] = div_fast(acc[j], __shfl_sync(0xffffffffu, s_tok, j), __shfl_sync(0xffffffffu, r_tok, j),
                                          __shfl_sync(0xffffffffu, k_tok, j));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[j] = __fdiv_rn(acc[j], __shfl_sync(0xffffffffu, s_tok, j));
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const uint32_t codes = e4m3x2(acc[j], acc[j + 1]);
                    if (j < ti.rows) p.hq[(size_t)(ti.row0 + j) * p.ldq + n] = (uint8_t)(codes & 0xffu);
                    if (j + 1 < ti.rows) p.hq[(size_t)(ti.row0 + j + 1) * p.ldq + n] = (uint8_t)(codes >> 8);
                }
            } else {
                const int slot_l = reinterpret_cast<const int*>(m)[M.slot + lane];
                const float w_l = m[M.w + lane];
                mbar_arrive(smem_u32(&mempty_bar[slot]));
                const bool two = ti.two;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int slot_t = __shfl_sync(0xffffffffu, slot_l, j);
                    const float w = __shfl_sync(0xffffffffu, w_l, j);
                    if (j < ti.rows) {
                        p.part[(size_t)slot_t * p.ldp + n] = w * acc[j];
                        if (C::TWO && two) p.part[(size_t)slot_t * p.ldp + n + p.up_rows] = w * acc[C::BT + j];
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

// The stage ring takes the shared memory the metadata slots and the kernel's
// static arrays leave, up to `max_stages` stages.
template <bool GATED, bool PAIRED>
static cudaError_t launch_dec(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p, int grid,
                              int max_stages, cudaStream_t st) {
    using C = DecCfg<GATED, PAIRED>;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, moe_gemm_decode_kernel<GATED, PAIRED>);
    if (e != cudaSuccess) return e;
    const size_t meta = (size_t)2 * dec_meta(p.KB).floats * 4;
    const long long room = (long long)optin - (long long)fa.sharedSizeBytes - 1024 - (long long)meta;
    int nst = (int)(room / C::STAGE_BYTES);
    if (nst > max_stages) nst = max_stages;
    if (nst > C::MAX_STAGES) nst = C::MAX_STAGES;
    if (nst < 2) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)nst * C::STAGE_BYTES + meta + 1024;
    e = cudaFuncSetAttribute(moe_gemm_decode_kernel<GATED, PAIRED>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(moe_gemm_decode_kernel<GATED, PAIRED>, dim3(grid), dim3(C::THREADS), smem, st, tmW, tmX, p, nst);
}

cudaError_t launch_gemm_gateup_decode(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p, int grid,
                                      cudaStream_t st) {
    return launch_dec<true, false>(tmW, tmX, p, grid, kDecStagesGateUp, st);
}

cudaError_t launch_gemm_down_decode(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p, int grid,
                                    cudaStream_t st) {
    // up_rows != 0: tiles of two w2 row blocks (the tile list was counted with
    // ceil(row blocks / 2) n-tiles per m-tile)
    return p.up_rows != 0 ? launch_dec<false, true>(tmW, tmX, p, grid, kDecStagesGateUp, st)
                          : launch_dec<false, false>(tmW, tmX, p, grid, kDecStagesDown, st);
}

}  // namespace moe
