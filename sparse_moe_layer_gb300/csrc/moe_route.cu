// Routing side of the sparse MoE layer ("GPT-OSS on Day 0", perplexity.ai hub
// blog): router GEMV + top-k + softmax over the selected k, the grouping of
// tokens by expert (dispatch), 1x128 FP8 quantisation of x, and the weighted
// combine back to token order.  Also the 128x128 block packer for weights and
// the stand-alone 1x128 quantiser.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// ===================================================================== router
// a1 + a2 + the histogram half of a3.  logits[t,e] = sum_h x[t,h]*Wr[e,h] +
// br[e] with bf16 inputs and fp32 accumulation; the k largest (ties -> lower
// expert index) are stored in ascending expert order with the softmax over
// their k logits in fp32 ("softmax after top-k", "softmax only over the
// selected experts"), rounded to bf16 for the combine ("expert weights in
// bfloat16").  One kernel computes the logits and selects (router_kernel: a
// thread-block cluster per token tile; router_tc_kernel: tensor cores, for
// large batches); the last CTA of either turns the (chunk, expert) histogram
// into the per-expert row offsets, per-chunk row bases and GEMM tile lists,
// so those are final when the router grid completes.

// The k largest of lg[0..E) for one warp (ties -> lower index), ascending.
__device__ __forceinline__ void select_topk(const float* lg, int E, int k, int lane, int* chosen) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? lg[e] : -INFINITY;
    }
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        chosen[j] = be;
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
    }
    for (int a = 1; a < k; ++a) {
        const int key = chosen[a];
        int b = a - 1;
        while (b >= 0 && chosen[b] > key) {
            chosen[b + 1] = chosen[b];
            --b;
        }
        chosen[b + 1] = key;
    }
}

// Softmax over the chosen logits (fp32, slot order) and the token's outputs;
// lane j < k writes slot j and counts it in the histogram.
__device__ __forceinline__ void write_route(const RouteParams& p, int t, const float* lg, const int* chosen,
                                            int lane) {
    float m = -INFINITY;
    for (int j = 0; j < p.k; ++j) m = fmaxf(m, lg[chosen[j]]);
    float z = 0.f;
    for (int j = 0; j < p.k; ++j) z += expf(lg[chosen[j]] - m);
    if (lane < p.k) {
        int e = chosen[0];
#pragma unroll
        for (int j = 1; j < kMaxTopK; ++j)
            if (j == lane) e = chosen[j];
        const float w = expf(lg[e] - m) / z;
        p.topk_idx[(size_t)t * p.k + lane] = e;
        p.topk_w[(size_t)t * p.k + lane] = w;
        __nv_bfloat16 wb = __float2bfloat16_rn(w);
        p.topk_wb[(size_t)t * p.k + lane] = *reinterpret_cast<uint16_t*>(&wb);
        atomicAdd(&p.hist[(size_t)(t / kChunkTokens) * p.E + e], 1);
    }
}

// Run by the last CTA (blockDim 256): counts, offsets, chunk bases, tile lists.
// The (chunk, expert) histogram is first copied into `buf` (the CTA's shared
// memory, free by then) with coalesced loads when it fits in `cap` ints, so
// the per-expert sums over the chunks run from shared memory instead of one
// dependent L2 round trip per chunk.
__device__ void finish_scan(const RouteParams& p, int* buf, int cap) {
    __shared__ int s_count[kMaxExperts], s_off[kMaxExperts];
    const int n = p.nchunks * p.E;
    const bool staged = n <= cap;
    if (staged)
        for (int i = threadIdx.x; i < n; i += blockDim.x) buf[i] = __ldcg(&p.hist[i]);
    __syncthreads();
    auto h = [&](int c, int e) { return staged ? buf[(size_t)c * p.E + e] : __ldcg(&p.hist[(size_t)c * p.E + e]); };
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        int run = 0;
        for (int c = 0; c < p.nchunks; ++c) run += h(c, e);
        s_count[e] = run;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // exclusive scans of the counts and of the m-tiles over the experts by
        // one warp: lane l owns experts [8l, 8l+8) (E <= 256)
        const int lane = threadIdx.x;
        int cnt[8], mt[8];
        int tc = 0, tm = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            cnt[i] = e < p.E ? s_count[e] : 0;
            mt[i] = (cnt[i] + p.bm - 1) / p.bm;
            tc += cnt[i];
            tm += mt[i];
        }
        int ic = tc, im = tm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vc = __shfl_up_sync(0xffffffffu, ic, o);
            const int vm = __shfl_up_sync(0xffffffffu, im, o);
            if (lane >= o) {
                ic += vc;
                im += vm;
            }
        }
        int off = ic - tc, mts = im - tm;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < p.E) {
                s_off[e] = off;
                p.offset[e] = off;
                p.count[e] = cnt[i];
                p.tiles1[e] = mts * p.nt1;
                p.tiles2[e] = mts * p.nt2;
            }
            off += cnt[i];
            mts += mt[i];
        }
        if (lane == 31) {
            p.offset[p.E] = off;
            p.tiles1[p.E] = mts * p.nt1;
            p.tiles2[p.E] = mts * p.nt2;
            p.status[kStatusTiles1] = (uint32_t)(mts * p.nt1);
            p.status[kStatusTiles2] = (uint32_t)(mts * p.nt2);
            p.status[kStatusTileRows] = (uint32_t)p.bm;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        int run = s_off[e];
        for (int c = 0; c < p.nchunks; ++c) {
            p.chunk_base[(size_t)c * p.E + e] = run;
            run += h(c, e);
        }
    }
}

// True in every thread of the CTA that is the `total`-th to arrive on *ctr.
// The barrier orders every thread's earlier writes before thread 0's
// GPU-scope fence, which (fences are cumulative) orders them before its
// count; in the last CTA thread 0 fences again after the count, and the
// barrier behind it orders the other threads' reads after that.
__device__ __forceinline__ bool last_to_arrive(int* ctr, int total) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const bool last = atomicAdd(ctr, 1) == total - 1;
        if (last) __threadfence();
        s_last = last;
    }
    __syncthreads();
    return s_last != 0;
}

// ---- router: a token tile x all experts per cluster, K split over its CTAs ----
// A cluster of KS CTAs owns a tile of TOK tokens (32 for decode-sized batches,
// 128 -- 64 beyond 128 experts -- for large ones, so that each tile reads the
// router weights once for more tokens); CTA r of it accumulates the
// logits of all experts over its own run of 64-wide K chunks on bf16 mma.sync
// (fp32 accumulation), with kRtNB chunks of x and router weights in flight.
// The KS partial tiles are then summed in rank order through distributed
// shared memory (the same order whatever CTA sums), each CTA finishing the
// tokens r, r + KS, ...: bias, top-k and softmax for one token per warp.  So
// small batches spread over up to 8x (16x with at most 64 experts) more SMs
// than they have token tiles, and no partial logit goes through global memory.
constexpr int kRtTok = 32;      // tokens per cluster, decode-sized batches
constexpr int kRtTokBig = 128;  // tokens per cluster, large batches (64 beyond 128 experts)
constexpr int kRtBigT = 2048;   // batches of at least this many tokens take the large tile
constexpr int kRtK = 64;    // K chunk
constexpr int kRtLd = 72;   // padded smem row (bf16 elements): conflict-free fragment loads
constexpr int kRtNB = 4;    // chunks in flight per CTA

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NTW, int TOK>
struct RouterCfg {
    static constexpr int EP = 64 * NTW;                   // experts padded to 8 warps x NTW n8 tiles
    static constexpr int CHUNK = (TOK + EP) * kRtLd;      // bf16 elements of one staged K chunk
    static constexpr int LDL = EP + 4;                    // fp32 row of a logit tile
    static constexpr size_t LOAD_BYTES = (size_t)kRtNB * CHUNK * 2;
    static constexpr size_t TILE_BYTES = (size_t)2 * TOK * LDL * 4;  // partial + finished logits
    static constexpr size_t SMEM = LOAD_BYTES > TILE_BYTES ? LOAD_BYTES : TILE_BYTES;
};

// cpc: K chunks per CTA.  VEC: H % 8 == 0 (16-byte cp.async rows).
template <int NTW, bool VEC, int TOK>
__global__ void __launch_bounds__(256) router_kernel(RouteParams p, int cpc) {
    using C = RouterCfg<NTW, TOK>;
    constexpr int MT = TOK / 16;  // m16 tiles of tokens (every warp covers all of them)
    constexpr int EP = C::EP, LDL = C::LDL;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* cbuf = reinterpret_cast<uint16_t*>(smem);  // [kRtNB][(kRtTok + EP) * kRtLd]
    const uint32_t rank = cluster_ctarank(), KS = cluster_nctarank();
    const int t0 = (int)cluster_id_x() * TOK;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int nchunk = (p.H + kRtK - 1) / kRtK;
    const int c0 = (int)rank * cpc;
    const int nmine = max(0, min(cpc, nchunk - c0));

    auto load_chunk = [&](int ch, int buf) {
        uint16_t* xs = cbuf + buf * C::CHUNK;  // [TOK][kRtLd] then [EP][kRtLd]
        const int k0 = ch * kRtK;
        if (VEC) {
            for (int i = tid; i < (TOK + EP) * 8; i += 256) {
                const int r = i >> 3, q = i & 7, k = k0 + q * 8;
                const bool isx = r < TOK;
                const int row = isx ? t0 + r : r - TOK;
                const bool ok = (isx ? row < p.T : row < p.E) && k < p.H;
                const uint16_t* src = isx ? p.x + (size_t)row * p.H + k : p.rw + (size_t)row * p.H + k;
                cp_async16(smem_u32(xs + r * kRtLd + q * 8), ok ? src : p.x, ok);
            }
        } else {
            for (int i = tid; i < (TOK + EP) * kRtK; i += 256) {
                const int r = i / kRtK, q = i - r * kRtK, k = k0 + q;
                const bool isx = r < TOK;
                const int row = isx ? t0 + r : r - TOK;
                const bool ok = (isx ? row < p.T : row < p.E) && k < p.H;
                xs[r * kRtLd + q] = ok ? (isx ? p.x[(size_t)row * p.H + k] : p.rw[(size_t)row * p.H + k]) : (uint16_t)0;
            }
        }
    };

    float acc[MT][NTW][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;

    // kRtNB chunks in flight; one commit group per chunk slot (empty past the end)
#pragma unroll
    for (int i = 0; i < kRtNB; ++i) {
        if (i < nmine) load_chunk(c0 + i, i);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int i = 0; i < nmine; ++i) {
        const int buf = i % kRtNB;
        asm volatile("cp.async.wait_group %0;" ::"n"(kRtNB - 1) : "memory");
        __syncthreads();
        const uint16_t* xb = cbuf + buf * C::CHUNK;
        const uint16_t* wb = xb + TOK * kRtLd;
#pragma unroll
        for (int ks = 0; ks < kRtK / 16; ++ks) {
            const int kk = ks * 16 + 2 * c;
            uint32_t a[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint16_t* r0 = xb + (m * 16 + g) * kRtLd;
                const uint16_t* r1 = r0 + 8 * kRtLd;
                a[m][0] = *reinterpret_cast<const uint32_t*>(r0 + kk);
                a[m][1] = *reinterpret_cast<const uint32_t*>(r1 + kk);
                a[m][2] = *reinterpret_cast<const uint32_t*>(r0 + kk + 8);
                a[m][3] = *reinterpret_cast<const uint32_t*>(r1 + kk + 8);
            }
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const uint16_t* br = wb + ((warp * NTW + j) * 8 + g) * kRtLd;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(br + kk);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(br + kk + 8);
#pragma unroll
                for (int m = 0; m < MT; ++m) mma_bf16_16816(acc[m][j], a[m], b0, b1);
            }
        }
        __syncthreads();
        if (i + kRtNB < nmine) load_chunk(c0 + i + kRtNB, buf);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();

    // this CTA's partial logits (no bias) into shared memory, visible to the cluster
    float* part = reinterpret_cast<float*>(smem);  // [TOK][LDL]
    float* lg = part + TOK * LDL;                   // [ceil(TOK / KS)][LDL]
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < NTW; ++j) {
            const int col = (warp * NTW + j) * 8 + 2 * c;
            const int row = m * 16 + g;
            part[row * LDL + col] = acc[m][j][0];
            part[row * LDL + col + 1] = acc[m][j][1];
            part[(row + 8) * LDL + col] = acc[m][j][2];
            part[(row + 8) * LDL + col + 1] = acc[m][j][3];
        }
    cluster_sync_all();
    // tokens rank, rank + KS, ...: sum the KS partials in rank order, add the bias
    const int nmy = (TOK - (int)rank + (int)KS - 1) / (int)KS;
    for (int idx = tid; idx < nmy * EP; idx += 256) {
        const int li = idx / EP, e = idx - li * EP;
        const int r = (int)rank + li * (int)KS;
        const uint32_t a = smem_u32(part + r * LDL + e);
        float sum = 0.f;
        for (uint32_t q = 0; q < KS; ++q) sum += (q == rank) ? part[r * LDL + e] : ld_cluster_f32(a, q);
        lg[li * LDL + e] = e < p.E ? sum + bf16_bits_to_f32(p.rb[e]) : -INFINITY;
    }
    __syncthreads();
    for (int li = warp; li < nmy; li += 8) {
        const int t = t0 + (int)rank + li * (int)KS;
        if (t >= p.T) break;
        int chosen[kMaxTopK];
        select_topk(lg + li * LDL, p.E, p.k, lane, chosen);
        write_route(p, t, lg + li * LDL, chosen, lane);
    }
    // no CTA leaves while another may still read its partial tile
    cluster_sync_all();
    if (last_to_arrive(p.done, gridDim.x))
        finish_scan(p, reinterpret_cast<int*>(smem), (int)(C::SMEM / 4));
}

template <int NTW, bool VEC, int TOK>
static cudaError_t launch_router_t(const RouteParams& p, cudaStream_t st) {
    using C = RouterCfg<NTW, TOK>;
    const int ntiles = (p.T + TOK - 1) / TOK;
    const int nchunk = (p.H + kRtK - 1) / kRtK;
    // about two CTAs per SM in all with the small tile; one (shared memory)
    // with the large one
    const int want = TOK == kRtTok ? 296 : 152;
    // Up to 16 CTAs per cluster (a non-portable size) with at most 64 experts:
    // fewer K chunks per CTA shortened the router of a 64-token, 32-expert,
    // 2880-wide batch from 17.0-17.4 to 15.6-16.1 us, while 128 experts (a
    // longer rank-order sum per logit) gained nothing; 8 elsewhere, or where
    // this device cannot co-schedule 16.
    static std::atomic<int> wide_ok{-1};
    cudaError_t e = cudaFuncSetAttribute(router_kernel<NTW, VEC, TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    // function attributes belong to the current device's context: set on every launch
    const bool wide_attr =
        NTW == 1 &&
        cudaFuncSetAttribute(router_kernel<NTW, VEC, TOK>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess;
    if (!wide_attr) (void)cudaGetLastError();
    if (wide_attr && wide_ok.load() < 0) {
        int ok = 0;
        {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(16);
            q.blockDim = dim3(256);
            q.dynamicSmemBytes = C::SMEM;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 16;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, router_kernel<NTW, VEC, TOK>, &q) == cudaSuccess &&
                nclusters > 0)
                ok = 1;
            else
                (void)cudaGetLastError();
        }
        wide_ok.store(ok);
    }
    const int ks_max = wide_attr && wide_ok.load() == 1 ? 16 : 8;
    int ks = ntiles >= want / 2 ? 1 : want / ntiles;
    ks = ks < 1 ? 1 : (ks > ks_max ? ks_max : ks);
    if (ks > nchunk) ks = nchunk;
    const int cpc = (nchunk + ks - 1) / ks;
    ks = (nchunk + cpc - 1) / cpc;  // no CTA without a chunk
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ntiles * ks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, router_kernel<NTW, VEC, TOK>, p, cpc);
}


template <int NTW, int TOK>
static cudaError_t launch_router_v(const RouteParams& p, cudaStream_t st) {
    return (p.H % 8) == 0 ? launch_router_t<NTW, true, TOK>(p, st) : launch_router_t<NTW, false, TOK>(p, st);
}

cudaError_t launch_router(const RouteParams& p, cudaStream_t st) {
    const bool big = p.T >= kRtBigT;
    if (p.E <= 64) return big ? launch_router_v<1, kRtTokBig>(p, st) : launch_router_v<1, kRtTok>(p, st);
    if (p.E <= 128) return big ? launch_router_v<2, kRtTokBig>(p, st) : launch_router_v<2, kRtTok>(p, st);
    return big ? launch_router_v<4, kRtTokBig / 2>(p, st) : launch_router_v<4, kRtTok>(p, st);
}

// ---- router on the tensor cores: large batches with 16-byte aligned rows ----
// One CTA per 128-token tile.  TMA brings 64-wide K chunks of the tile's x
// rows and of every router weight row (experts padded to NP, the padding
// zero-filled) into a ring; one thread issues tcgen05.mma kind::f16 (bf16 x
// bf16, fp32 accumulator in TMEM; M = 128 tokens, N = NP experts, K = 16 per
// instruction).  After the last chunk four warps each read the logits of 32
// tokens (TMEM lane = token), add the bias, keep the 8 largest in registers
// (ties -> lower expert index: experts are visited in ascending order and only
// a strictly larger logit moves ahead), and write the softmax over the first k
// of them in ascending expert order -- the same selection and arithmetic as
// the cluster kernel above, whose mma.sync path runs far below the tensor
// cores' rate on this part.
template <int NP>
struct RouterTcCfg {
    static constexpr int A_BYTES = 128 * 128;  // 128 tokens x 64 bf16
    static constexpr int B_BYTES = NP * 128;   // NP experts x 64 bf16
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = NP > 128 ? 4 : 6;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024;
    static constexpr int TMEM_COLS = NP < 32 ? 32 : NP;  // a power of two >= 32
    static constexpr uint32_t IDESC = idesc_bf16_f32(128, NP);
    static_assert(NP % 32 == 0 && NP <= 256, "expert padding");
};

template <int NP>
__global__ void __launch_bounds__(256, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const __grid_constant__ CUtensorMap tmW, RouteParams p) {
    using C = RouterTcCfg<NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full_bar[C::STAGES];
    __shared__ __align__(8) uint64_t empty_bar[C::STAGES];
    __shared__ __align__(8) uint64_t dfull_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float s_bias[NP];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * 128;
    const int nchunk = (p.H + 63) / 64;
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&dfull_bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), C::TMEM_COLS);
    for (int e = tid; e < NP; e += blockDim.x) s_bias[e] = e < p.E ? bf16_bits_to_f32(p.rb[e]) : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort_p = &abort_flag;
    uint32_t* err = p.status + kStatusError;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int c = 0;
            for (; c < nchunk; ++c) {
                const int stage = c % C::STAGES;
                const uint32_t phase = (uint32_t)(c / C::STAGES) & 1u;
                if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_p, err, kErrTimeoutProducer)) break;
                const uint32_t fb = smem_u32(&full_bar[stage]);
                mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
                const uint32_t a_dst = smem_u32(smem + stage * C::STAGE_BYTES);
                tma_load_2d(a_dst, &tmX, c * 64, t0, fb);
                tma_load_2d(a_dst + C::A_BYTES, &tmW, c * 64, 0, fb);
            }
            // the last fill of every stage has landed before the CTA may exit
            int dummy = 0;
            for (int q = max(0, c - C::STAGES); q < c; ++q)
                mbar_wait(smem_u32(&full_bar[q % C::STAGES]), (uint32_t)(q / C::STAGES) & 1u, &dummy, err,
                          kErrTimeoutProducer);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            for (int c = 0; c < nchunk; ++c) {
                const int stage = c % C::STAGES;
                if (!mbar_wait(smem_u32(&full_bar[stage]), (uint32_t)(c / C::STAGES) & 1u, abort_p, err,
                               kErrTimeoutMma))
                    break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(smem + stage * C::STAGE_BYTES);
                const uint32_t b_base = a_base + C::A_BYTES;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    mma_bf16(tmem, smem_desc_sw128(a_base + 32 * k4), smem_desc_sw128(b_base + 32 * k4), C::IDESC,
                             (c | k4) != 0 ? 1u : 0u);
                mma_commit(smem_u32(&empty_bar[stage]));
            }
            // the accumulator is complete (or, after an abort, every issued MMA has
            // finished) once this commit lands
            mma_commit(smem_u32(&dfull_bar));
            int dummy = 0;
            mbar_wait(smem_u32(&dfull_bar), 0, &dummy, err, kErrTimeoutMma);
        }
    } else if (warp >= 4) {
        // ------------------------------------------ selection + softmax
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        const int t = t0 + row;
        const bool ok = mbar_wait(smem_u32(&dfull_bar), 0, abort_p, err, kErrTimeoutEpilogue);
        tc_fence_after();
        if (ok) {
            float v[kMaxTopK];
            int id[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                v[j] = -INFINITY;
                id[j] = 0x7fffffff;
            }
            const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < NP; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(t_lane + (uint32_t)c0, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int e = c0 + i;
                    const float l = __uint_as_float(r[i]) + s_bias[e];
                    if (e < p.E && l > v[kMaxTopK - 1]) {
                        // insert, keeping v descending; an equal value stays behind
                        float cv = l;
                        int ci = e;
#pragma unroll
                        for (int j = 0; j < kMaxTopK; ++j) {
                            const bool gt = cv > v[j];
                            const float tv = v[j];
                            const int ti = id[j];
                            v[j] = gt ? cv : tv;
                            id[j] = gt ? ci : ti;
                            cv = gt ? tv : cv;
                            ci = gt ? ti : ci;
                        }
                    }
                }
            }
            if (t < p.T) {
                const int k = p.k;
                // the first k in ascending expert order (the rest sort behind them)
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j >= k) id[j] = 0x7fffffff;
#pragma unroll
                for (int a = 0; a < kMaxTopK; ++a)
#pragma unroll
                    for (int b = 0; b + 1 < kMaxTopK - a; ++b) {
                        const bool sw = id[b] > id[b + 1];
                        const int ib = id[b], ib1 = id[b + 1];
                        const float vb = v[b], vb1 = v[b + 1];
                        id[b] = sw ? ib1 : ib;
                        id[b + 1] = sw ? ib : ib1;
                        v[b] = sw ? vb1 : vb;
                        v[b + 1] = sw ? vb : vb1;
                    }
                float m = -INFINITY;
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j < k) m = fmaxf(m, v[j]);
                float z = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j < k) z += expf(v[j] - m);
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j) {
                    if (j < k) {
                        const float w = expf(v[j] - m) / z;
                        p.topk_idx[(size_t)t * k + j] = id[j];
                        p.topk_w[(size_t)t * k + j] = w;
                        __nv_bfloat16 wb = __float2bfloat16_rn(w);
                        p.topk_wb[(size_t)t * k + j] = *reinterpret_cast<uint16_t*>(&wb);
                        atomicAdd(&p.hist[(size_t)(t / kChunkTokens) * p.E + id[j]], 1);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    if (last_to_arrive(p.done, gridDim.x))
        finish_scan(p, reinterpret_cast<int*>(smem), C::STAGES * C::STAGE_BYTES / 4);
}

template <int NP>
static cudaError_t launch_router_tc_t(const RouteParams& p, const CUtensorMap& tmX, const CUtensorMap& tmW,
                                      cudaStream_t st) {
    using C = RouterTcCfg<NP>;
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    router_tc_kernel<NP><<<(p.T + 127) / 128, 256, C::SMEM, st>>>(tmX, tmW, p);
    return cudaGetLastError();
}

int router_tc_experts(int T, int H, int E) {
    // decode-sized batches stay on the cluster kernel: one CTA streaming the
    // router weights alone is slower than eight splitting K (oss20b_decode
    // router 15.7 us clustered, 24.9 us on one tensor-core CTA)
    if (T < kRtBigT || (H % 8) != 0 || E > 256) return 0;
    return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
}

cudaError_t launch_router_tc(const RouteParams& p, const CUtensorMap& tmX, const CUtensorMap& tmW, cudaStream_t st) {
    switch (router_tc_experts(p.T, p.H, p.E)) {
        case 32: return launch_router_tc_t<32>(p, tmX, tmW, st);
        case 64: return launch_router_tc_t<64>(p, tmX, tmW, st);
        case 128: return launch_router_tc_t<128>(p, tmX, tmW, st);
        case 256: return launch_router_tc_t<256>(p, tmX, tmW, st);
        default: return cudaErrorInvalidValue;
    }
}

// ======================================================= permute + x quant
// CTA = 8 warps over `tokens_per_cta` consecutive tokens (all in one 256-token
// chunk).  Row of (t, j) = chunk_base[chunk, e] + number of earlier tokens of
// the chunk routed to e, so rows are sorted by (expert, token).  Then every
// 128-group of the token is quantised (amax, s = amax/448, code = e4m3(x/s);
// one warp covers four groups) and written to each of the token's k rows.
__global__ void __launch_bounds__(256) permute_quant_kernel(PermuteParams p) {
    extern __shared__ __align__(16) uint8_t psm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(psm);  // this CTA's x rows, [tokens_per_cta][Hx]
    __shared__ int s_pre[kMaxExperts];
    __shared__ int s_base[kMaxExperts];
    __shared__ int s_idx[8 * kMaxTopK];
    __shared__ int s_row[8 * kMaxTopK];
    __shared__ int s_eoff[kMaxExperts];  // MXFP8: first row of each expert ...
    __shared__ int s_emt[kMaxExperts];   // ... and the m-tiles of the experts before it
    __shared__ long long s_aoff[8 * kMaxTopK];  // MXFP8: byte offset of each row's cell in K block 0's atom
    const int tpc = p.tokens_per_cta;
    const int t0 = blockIdx.x * tpc;
    const int chunk = t0 / kChunkTokens;
    const int c0 = chunk * kChunkTokens;
    const int nt = min(tpc, p.T - t0);
    const int Hx = (p.H + 7) & ~7;
    // x is an input of the layer, not an output of the router: stage it
    // before waiting for the router to finish
    if ((p.H & 7) == 0) {
        for (int i = threadIdx.x; i < nt * Hx / 8; i += blockDim.x)
            reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t0 * p.H) + i);
    } else {
        for (int i = threadIdx.x; i < nt * Hx; i += blockDim.x) {
            const int tt = i / Hx, h = i - tt * Hx;
            xs[i] = h < p.H ? p.x[(size_t)(t0 + tt) * p.H + h] : (uint16_t)0;
        }
    }
    pdl_wait();
    // The router has completed (its scan wrote the tile lists), so the gate/up
    // GEMM may be scheduled now: it reads those lists and streams its first
    // weight stages while this kernel quantises x, then waits for it.  Only
    // for a grid of one wave: the GEMM's CTAs would otherwise hold SMs that
    // this kernel's later CTAs need.
    if (p.early_dependents) pdl_allow_dependents();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_pre[e] = 0;
    // the router scanned the histogram: this chunk's first row of every expert
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        s_base[e] = p.chunk_base[(size_t)chunk * p.E + e];
        if (p.mx) {
            s_eoff[e] = p.offset[e];
            s_emt[e] = p.tiles1[e] / p.nt1;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < (t0 - c0) * p.k; i += blockDim.x) atomicAdd(&s_pre[p.topk_idx[(size_t)c0 * p.k + i]], 1);
    for (int i = threadIdx.x; i < nt * p.k; i += blockDim.x) s_idx[i] = p.topk_idx[(size_t)t0 * p.k + i];
    __syncthreads();
    for (int i = threadIdx.x; i < nt * p.k; i += blockDim.x) {
        int tt = i / p.k, j = i - tt * p.k, e = s_idx[i];
        int r = s_base[e] + s_pre[e];
        for (int u = 0; u < tt; ++u)
            for (int jj = 0; jj < p.k; ++jj) r += (s_idx[u * p.k + jj] == e);
        s_row[i] = r;
        if (p.mx) {
            const int local = r - s_eoff[e];
            const int mt = s_emt[e] + local / p.bm, m = local - (local / p.bm) * p.bm;
            s_aoff[i] = (long long)mt * (p.Hp / 128) * kMxAtomBytes + mx_atom_byte(m, 0);
        }
        int slot = (t0 + tt) * p.k + j;
        p.perm[r] = slot;
        p.inv[slot] = r;
    }
    __syncthreads();

    // One warp item = one token x 512 columns (four 128-groups): lane l holds
    // the 16 columns [16l, 16l+16) of the item, so lanes 8q..8q+7 hold group q
    // (MXFP8: lane pairs hold its four 1x32 groups), and writes them to each of
    // the token's k rows with one 16-byte store.
    const int G = p.Hp / 128;
    const int SG = (G + 3) / 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int item = warp; item < nt * SG; item += 8) {
        const int tt = item / SG, sg = item - tt * SG;
        const int g = sg * 4 + (lane >> 3);  // this lane's 128-group
        const int c = sg * 512 + lane * 16;  // its first column
        const bool act = g < G;              // lanes past the row's last group only join the shuffles
        float a[16];
        if (c + 16 <= Hx) {
            const uint4 v0 = *reinterpret_cast<const uint4*>(xs + tt * Hx + c);
            const uint4 v1 = *reinterpret_cast<const uint4*>(xs + tt * Hx + c + 8);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                a[2 * i] = __uint_as_float(w[i] << 16);
                a[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = (c + i < Hx) ? bf16_bits_to_f32(xs[tt * Hx + c + i]) : 0.f;
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(a[i]));
        uint4 q;
        uint32_t meta;  // MXFP8: the group's atom cell (four scale bytes); else the fp32 scale
        if (p.mx) {
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the lane pair's 32 values
            const uint32_t sb = mx_scale_byte(amax);
            const float inv = mx_inv_scale(sb);
            const uint32_t keep = mx_keep(amax);
            q.x = mx_quant4(a[0], a[1], a[2], a[3], inv, keep);
            q.y = mx_quant4(a[4], a[5], a[6], a[7], inv, keep);
            q.z = mx_quant4(a[8], a[9], a[10], a[11], inv, keep);
            q.w = mx_quant4(a[12], a[13], a[14], a[15], inv, keep);
            const int b = lane & ~7;
            meta = __shfl_sync(0xffffffffu, sb, b) | (__shfl_sync(0xffffffffu, sb, b + 2) << 8) |
                   (__shfl_sync(0xffffffffu, sb, b + 4) << 16) | (__shfl_sync(0xffffffffu, sb, b + 6) << 24);
        } else {
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float sc = group_scale(amax);
            const float rs = recip_rn(sc);
            q.x = quant4(a[0], a[1], a[2], a[3], amax, sc, rs);
            q.y = quant4(a[4], a[5], a[6], a[7], amax, sc, rs);
            q.z = quant4(a[8], a[9], a[10], a[11], amax, sc, rs);
            q.w = quant4(a[12], a[13], a[14], a[15], amax, sc, rs);
            meta = __float_as_uint(sc);
        }
        if (act) {
            const bool lead = (lane & 7) == 0;
            for (int j = 0; j < p.k; ++j) {
                const int r = s_row[tt * p.k + j];
                *reinterpret_cast<uint4*>(p.xq + (size_t)r * p.Hp + c) = q;
                if (lead) {
                    if (p.mx)
                        *reinterpret_cast<uint32_t*>(p.sxa + s_aoff[tt * p.k + j] + (size_t)g * kMxAtomBytes) = meta;
                    else
                        p.sx[(size_t)g * p.R + r] = __uint_as_float(meta);  // K-block-major [Hp/128, R]
                }
            }
        }
    }
}

cudaError_t launch_permute_quant(const PermuteParams& p_in, cudaStream_t st) {
    PermuteParams p = p_in;
    int grid = (p.T + p.tokens_per_cta - 1) / p.tokens_per_cta;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    p.early_dependents = grid <= sms ? 1 : 0;
    const size_t sm = (size_t)p.tokens_per_cta * ((p.H + 7) & ~7) * 2;
    cudaError_t e = cudaFuncSetAttribute(permute_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    return launch_pdl(permute_quant_kernel, dim3(grid), dim3(256), sm, st, p);
}

// ================================================================= combine
// out[t, n] = bf16_rn( sum_{j=0..k-1} part[t*k+j, n] ), slot order, fp32.
// ("Combine performs the weighted accumulation"; the weights were applied
// in the down GEMM's epilogue.)
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part, int T, int H, int ldp, int k,
                                                      uint16_t* __restrict__ out) {
    pdl_wait();
    const int n8 = (H + 7) / 8;
    const size_t total = (size_t)T * n8;
    const bool vec_out = (H & 7) == 0;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / n8);
        const int c = (int)(i - (size_t)t * n8) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const float4* src = reinterpret_cast<const float4*>(part + ((size_t)t * k + j) * ldp + c);
            float4 u = __ldcs(src), v = __ldcs(src + 1);
            acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
            acc[4] += v.x; acc[5] += v.y; acc[6] += v.z; acc[7] += v.w;
        }
        uint16_t o[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            __nv_bfloat16 b = __float2bfloat16_rn(acc[q]);
            o[q] = *reinterpret_cast<uint16_t*>(&b);
        }
        uint16_t* dst = out + (size_t)t * H + c;
        if (vec_out) {
            uint4 w;
            w.x = o[0] | ((uint32_t)o[1] << 16);
            w.y = o[2] | ((uint32_t)o[3] << 16);
            w.z = o[4] | ((uint32_t)o[5] << 16);
            w.w = o[6] | ((uint32_t)o[7] << 16);
            *reinterpret_cast<uint4*>(dst) = w;
        } else {
            for (int q = 0; q < 8 && c + q < H; ++q) dst[q] = o[q];
        }
    }
}

cudaError_t launch_combine(const float* part, int T, int H, int ldp, int k, uint16_t* out, int num_sms,
                           cudaStream_t st) {
    size_t total = (size_t)T * ((H + 7) / 8);
    size_t blocks = (total + 255) / 256;
    size_t cap = (size_t)num_sms * 8;
    int grid = (int)(blocks < cap ? blocks : cap);
    if (grid < 1) grid = 1;
    return launch_pdl(combine_kernel, dim3(grid), dim3(256), 0, st, part, T, H, ldp, k, out);
}

// ============================================================ weight packer
// One CTA per (128x128 destination block, expert); blocks are stored
// contiguously (16 KB each, [E][row block][K block][128][128]) so the GEMMs
// stream every weight tile as one contiguous 16 KB read.  Destination row dr maps
// to a source row: gated_I > 0 (w13): gate rows [0,I) -> [0,I), up rows
// [I,2I) -> [Ip, Ip+I); gated_I == 0 (w2): identity.  Rows/columns beyond
// the source are zero pad.  s = amax/448 (1 for an all-zero block), code =
// e4m3(w/s).
__global__ void __launch_bounds__(256) pack_blocks_kernel(const float* __restrict__ src, int rows_src, int cols,
                                                          int rows_p, int cols_p, int gated_I, uint8_t* __restrict__ q,
                                                          float* __restrict__ s) {
    const int bj = blockIdx.x, bi = blockIdx.y, e = blockIdx.z;
    const int r_local = threadIdx.x >> 1;
    const int dr = bi * 128 + r_local;
    const int c0 = bj * 128 + (threadIdx.x & 1) * 64;
    int sr;
    if (gated_I > 0) {
        const int Ip = rows_p / 2;
        sr = dr < Ip ? (dr < gated_I ? dr : -1) : (dr - Ip < gated_I ? gated_I + dr - Ip : -1);
    } else {
        sr = dr < rows_src ? dr : -1;
    }
    const float* row = sr >= 0 ? src + ((size_t)e * rows_src + sr) * cols : nullptr;
    float v[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = (row && c0 + i < cols) ? __ldg(row + c0 + i) : 0.f;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float s_red[8];
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = s_red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_red[w]);
    const float sc = group_scale(amax);
    const float rc = recip_rn(sc);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) packed[i] = quant4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], amax, sc, rc);
    // blocked layout: block (e, bi, bj) is 16 KB contiguous, row-major inside
    const size_t blk = ((size_t)e * (rows_p / 128) + bi) * (cols_p / 128) + bj;
    uint4* dst = reinterpret_cast<uint4*>(q + blk * 16384 + (size_t)r_local * 128 + (threadIdx.x & 1) * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    if (threadIdx.x == 0) s[((size_t)e * (rows_p / 128) + bi) * (cols_p / 128) + bj] = sc;
}

cudaError_t launch_pack_blocks(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p, int gated_I,
                               uint8_t* q, float* s, cudaStream_t st) {
    dim3 grid(cols_p / 128, rows_p / 128, E);
    pack_blocks_kernel<<<grid, 256, 0, st>>>(src, rows_src, cols, rows_p, cols_p, gated_I, q, s);
    return cudaGetLastError();
}

// Row-major codes [E, rows, cols] -> blocked [E, rows/128, cols/128, 128, 128]
// (each 128x128 block 16 KB contiguous, row-major inside): one CTA per block,
// a thread moves 64 bytes of one row with 16-byte loads and stores.
__global__ void __launch_bounds__(256) block_codes_kernel(const uint8_t* __restrict__ src, int rows, int cols,
                                                          uint8_t* __restrict__ dst) {
    const int bj = blockIdx.x, bi = blockIdx.y, e = blockIdx.z;
    const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
    const uint4* in =
        reinterpret_cast<const uint4*>(src + ((size_t)e * rows + (size_t)bi * 128 + r) * cols + bj * 128 + h * 64);
    const size_t blk = ((size_t)e * (rows / 128) + bi) * (cols / 128) + bj;
    uint4* out = reinterpret_cast<uint4*>(dst + blk * 16384 + (size_t)r * 128 + h * 64);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(in + i);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = v[i];
}

cudaError_t launch_block_codes(const uint8_t* src, int E, int rows, int cols, uint8_t* dst, cudaStream_t st) {
    dim3 grid(cols / 128, rows / 128, E);
    block_codes_kernel<<<grid, 256, 0, st>>>(src, rows, cols, dst);
    return cudaGetLastError();
}

// ============================================== stand-alone 1x128 quantiser
__global__ void __launch_bounds__(256) quantize_rows_kernel(const float* __restrict__ in, int rows, int cols, int ld_in,
                                                            uint8_t* __restrict__ q, float* __restrict__ s) {
    const int G = (cols + 127) / 128;
    const int cp = G * 128;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (long item = warp; item < (long)rows * G; item += nwarps) {
        const int r = (int)(item / G), g = (int)(item - (long)r * G);
        const int c = g * 128 + lane * 4;
        float a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = (c + i < cols) ? in[(size_t)r * ld_in + c + i] : 0.f;
        float amax = fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = group_scale(amax);
        *reinterpret_cast<uint32_t*>(q + (size_t)r * cp + c) = quant4(a[0], a[1], a[2], a[3], amax, sc, recip_rn(sc));
        if (lane == 0) s[(size_t)r * G + g] = sc;
    }
}

cudaError_t launch_quantize_rows(const float* in, int rows, int cols, int ld_in, uint8_t* q, float* s,
                                 cudaStream_t st) {
    long items = (long)rows * ((cols + 127) / 128);
    long blocks = (items + 7) / 8;
    int grid = (int)(blocks < 4096 ? blocks : 4096);
    if (grid < 1) grid = 1;
    quantize_rows_kernel<<<grid, 256, 0, st>>>(in, rows, cols, ld_in, q, s);
    return cudaGetLastError();
}

// ======================================================= MXFP8 weight packer
// Same blocks and row mapping as pack_blocks_kernel; every weight row is
// quantised along K in groups of 32 (mx_scale_byte / mx_quant4), and the
// block's 128 rows x 4 groups of scale bytes form one 512-byte atom
// (mx_atom_byte), stored [E][row block][K block][512] beside the codes.
__global__ void __launch_bounds__(256) pack_blocks_mx_kernel(const float* __restrict__ src, int rows_src, int cols,
                                                             int rows_p, int cols_p, int gated_I,
                                                             uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    const int bj = blockIdx.x, bi = blockIdx.y, e = blockIdx.z;
    const int r_local = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int dr = bi * 128 + r_local;
    const int c0 = bj * 128 + half * 64;
    int sr;
    if (gated_I > 0) {
        const int Ip = rows_p / 2;
        sr = dr < Ip ? (dr < gated_I ? dr : -1) : (dr - Ip < gated_I ? gated_I + dr - Ip : -1);
    } else {
        sr = dr < rows_src ? dr : -1;
    }
    const float* row = sr >= 0 ? src + ((size_t)e * rows_src + sr) * cols : nullptr;
    const size_t blk = ((size_t)e * (rows_p / 128) + bi) * (cols_p / 128) + bj;
    uint32_t packed[16];
    uint32_t bytes = 0;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        float v[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = c0 + 32 * g + i;
            v[i] = (row && c < cols) ? __ldg(row + c) : 0.f;
            amax = fmaxf(amax, fabsf(v[i]));
        }
        const uint32_t sb = mx_scale_byte(amax);
        const float inv = mx_inv_scale(sb);
        const uint32_t keep = mx_keep(amax);
#pragma unroll
        for (int i = 0; i < 8; ++i) packed[8 * g + i] = mx_quant4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], inv, keep);
        bytes |= sb << (8 * g);
    }
    uint4* dst = reinterpret_cast<uint4*>(q + blk * 16384 + (size_t)r_local * 128 + half * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    *reinterpret_cast<uint16_t*>(s + blk * kMxAtomBytes + mx_atom_byte(r_local, 2 * half)) = (uint16_t)bytes;
}

cudaError_t launch_pack_blocks_mx(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p, int gated_I,
                                  uint8_t* q, uint8_t* s, cudaStream_t st) {
    dim3 grid(cols_p / 128, rows_p / 128, E);
    pack_blocks_mx_kernel<<<grid, 256, 0, st>>>(src, rows_src, cols, rows_p, cols_p, gated_I, q, s);
    return cudaGetLastError();
}

// ============================================== MXFP4 weight packer
// OCP MX v1.0 with FP4 E2M1 elements (section 5.3.3): magnitudes 0, 0.5, 1,
// 1.5, 2, 3, 4, 6 (codes 0-7), the sign in bit 3, no infinities or NaN.
// Nearest value, ties to the even code (the midpoints 0.25, 1.25, 2.5 and 5
// round down, 0.75, 1.75 and 3.5 up), magnitudes above 6 saturate to 6; the
// sign of v is kept where it rounds to 0.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
    const float a = fabsf(v);
    const uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                       (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
    return c | ((__float_as_uint(v) >> 28) & 8u);
}

// Shared exponent of a 32-group (section 6.3): X = floor(log2(amax)) - 2 (2 =
// the exponent of E2M1's largest normal, 6 = 1.5 * 2^2), clamped to [-127,
// 127], stored as X + 127; for a normal amax with biased fp32 exponent b that
// is b - 2, every amax below 2^-125 lands on the clamp (byte 0), and an
// all-zero group gets byte 0 with +0 codes.
__device__ __forceinline__ uint32_t mx4_scale_byte(float amax) {
    const int b = (int)((__float_as_uint(amax) >> 23) & 0xffu);
    return amax == 0.0f ? 0u : (uint32_t)max(b - 2, 0);
}

// fp32 masters -> blocked E2M1 codes, two per byte (value 2j in the low
// nibble of byte j), one 128 x 64-byte block per (row block, K block), and the
// same 512-byte scale atoms as the MXFP8 packer.  Thread layout as
// pack_blocks_mx_kernel: two threads per row, 64 columns (two groups) each.
__global__ void __launch_bounds__(256) pack_blocks_mx4_kernel(const float* __restrict__ src, int rows_src, int cols,
                                                              int rows_p, int cols_p, int gated_I,
                                                              uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    const int bj = blockIdx.x, bi = blockIdx.y, e = blockIdx.z;
    const int r_local = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int dr = bi * 128 + r_local;
    const int c0 = bj * 128 + half * 64;
    int sr;
    if (gated_I > 0) {
        const int Ip = rows_p / 2;
        sr = dr < Ip ? (dr < gated_I ? dr : -1) : (dr - Ip < gated_I ? gated_I + dr - Ip : -1);
    } else {
        sr = dr < rows_src ? dr : -1;
    }
    const float* row = sr >= 0 ? src + ((size_t)e * rows_src + sr) * cols : nullptr;
    const size_t blk = ((size_t)e * (rows_p / 128) + bi) * (cols_p / 128) + bj;
    uint32_t packed[8];
    uint32_t bytes = 0;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        float v[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = c0 + 32 * g + i;
            v[i] = (row && c < cols) ? __ldg(row + c) : 0.f;
            amax = fmaxf(amax, fabsf(v[i]));
        }
        const uint32_t sb = mx4_scale_byte(amax);
        const float inv = mx_inv_scale(sb);
        const uint32_t keep = mx_keep(amax);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) word |= e2m1_code(mx_scaled(v[8 * w + i], inv, keep)) << (4 * i);
            packed[4 * g + w] = word;
        }
        bytes |= sb << (8 * g);
    }
    uint4* dst = reinterpret_cast<uint4*>(q + blk * 8192 + (size_t)r_local * 64 + half * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    *reinterpret_cast<uint16_t*>(s + blk * kMxAtomBytes + mx_atom_byte(r_local, 2 * half)) = (uint16_t)bytes;
}

cudaError_t launch_pack_blocks_mx4(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p,
                                   int gated_I, uint8_t* q, uint8_t* s, cudaStream_t st) {
    dim3 grid(cols_p / 128, rows_p / 128, E);
    pack_blocks_mx4_kernel<<<grid, 256, 0, st>>>(src, rows_src, cols, rows_p, cols_p, gated_I, q, s);
    return cudaGetLastError();
}

// ============================================== stand-alone 1x32 quantiser
// fp32 [rows, cols] -> codes [rows, cp], scale bytes [rows, cp/32] (row-major,
// cp = cols padded to 128); one warp per 128-wide block, 8 lanes per group.
__global__ void __launch_bounds__(256) quantize_rows_mx_kernel(const float* __restrict__ in, int rows, int cols,
                                                               int ld_in, uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ s) {
    const int G = (cols + 127) / 128;
    const int cp = G * 128;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (long item = warp; item < (long)rows * G; item += nwarps) {
        const int r = (int)(item / G), g = (int)(item - (long)r * G);
        const int c = g * 128 + lane * 4;
        float a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = (c + i < cols) ? in[(size_t)r * ld_in + c + i] : 0.f;
        float amax = fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3])));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const uint32_t sb = mx_scale_byte(amax);
        *reinterpret_cast<uint32_t*>(q + (size_t)r * cp + c) =
            mx_quant4(a[0], a[1], a[2], a[3], mx_inv_scale(sb), mx_keep(amax));
        if ((lane & 7) == 0) s[(size_t)r * (cp / 32) + g * 4 + (lane >> 3)] = (uint8_t)sb;
    }
}

cudaError_t launch_quantize_rows_mx(const float* in, int rows, int cols, int ld_in, uint8_t* q, uint8_t* s,
                                    cudaStream_t st) {
    long items = (long)rows * ((cols + 127) / 128);
    long blocks = (items + 7) / 8;
    int grid = (int)(blocks < 4096 ? blocks : 4096);
    if (grid < 1) grid = 1;
    quantize_rows_mx_kernel<<<grid, 256, 0, st>>>(in, rows, cols, ld_in, q, s);
    return cudaGetLastError();
}

// ================================================ bounded-wait self check
__global__ void bounded_wait_kernel(uint64_t timeout_ns, int arrivals, uint32_t* result) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    abort_flag = 0;
    mbar_init(b, 1);
    fence_barrier_init();
    if (arrivals > 0) mbar_arrive(b);
    const bool ok = mbar_wait(b, 0, &abort_flag, nullptr, 0u, timeout_ns);
    *result = ok ? 1u : 2u;
}

cudaError_t launch_bounded_wait_test(uint64_t timeout_ns, int arrivals, uint32_t* result, cudaStream_t st) {
    bounded_wait_kernel<<<1, 32, 0, st>>>(timeout_ns, arrivals, result);
    return cudaGetLastError();
}

}  // namespace moe
