// Routing side of the sparse MoE layer ("GPT-OSS on Day 0", perplexity.ai hub
// blog): router GEMV + top-k + softmax over the selected k, the grouping of
// tokens by expert (dispatch), 1x128 FP8 quantisation of x, and the weighted
// combine back to token order.  Also the 128x128 block packer for weights and
// the stand-alone 1x128 quantiser.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// ===================================================================== router
// One CTA (8 warps) per TPB tokens.  The tokens' x rows sit in shared memory;
// warp w computes the logits of experts w, w+8, ... for all TPB tokens (each
// router_w row is read once per CTA), fp32 accumulation of bf16 products.
// Then warp j (< TPB) selects token j's top-k (ties -> lower expert index),
// stores the k experts in ascending order with the softmax over their k
// logits (fp32, "softmax after top-k" / "softmax only over the selected
// experts", weights rounded to bf16), and counts them in the (chunk, expert)
// histogram.  The last CTA to finish turns the histogram into per-expert
// row offsets, per-chunk row bases and the GEMM tile lists.
template <int TPB>
__global__ void __launch_bounds__(256) router_kernel(RouteParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int Hx = (p.H + 7) & ~7;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    float* lg = reinterpret_cast<float*>(smem + (size_t)TPB * Hx * 2);
    const int t0 = blockIdx.x * TPB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < TPB * Hx; i += 256) {
        int tt = i / Hx, h = i - tt * Hx, t = t0 + tt;
        xs[i] = (t < p.T && h < p.H) ? p.x[(size_t)t * p.H + h] : (uint16_t)0;
    }
    __syncthreads();

    const bool vec = (p.H & 7) == 0;
    for (int e = warp; e < p.E; e += 8) {
        float acc[TPB];
#pragma unroll
        for (int tt = 0; tt < TPB; ++tt) acc[tt] = 0.f;
        const uint16_t* wr = p.rw + (size_t)e * p.H;
        for (int h = lane * 8; h < Hx; h += 256) {
            float w[8];
            if (vec) {
                uint4 v = __ldg(reinterpret_cast<const uint4*>(wr + h));
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    w[2 * i] = __uint_as_float(u[i] << 16);
                    w[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = (h + i < p.H) ? bf16_bits_to_f32(wr[h + i]) : 0.f;
            }
#pragma unroll
            for (int tt = 0; tt < TPB; ++tt) {
                uint4 v = *reinterpret_cast<const uint4*>(xs + tt * Hx + h);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[tt] = fmaf(__uint_as_float(u[i] << 16), w[2 * i], acc[tt]);
                    acc[tt] = fmaf(__uint_as_float(u[i] & 0xffff0000u), w[2 * i + 1], acc[tt]);
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < TPB; ++tt) {
            float v = acc[tt];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[tt] = v;
        }
        if (lane == 0) {
            const float b = bf16_bits_to_f32(p.rb[e]);
#pragma unroll
            for (int tt = 0; tt < TPB; ++tt) lg[tt * p.E + e] = acc[tt] + b;
        }
    }
    __syncthreads();

    if (warp < TPB && t0 + warp < p.T) {
        const int t = t0 + warp;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int e = lane + 32 * i;
            v[i] = e < p.E ? lg[warp * p.E + e] : -INFINITY;
        }
        uint32_t taken = 0;
        int chosen[kMaxTopK];
        for (int j = 0; j < p.k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int e = lane + 32 * i;
                if (e < p.E && !((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                    bv = ov;
                    be = oe;
                }
            }
            chosen[j] = be;
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
        }
        // ascending expert order
        for (int a = 1; a < p.k; ++a) {
            int key = chosen[a], b = a - 1;
            while (b >= 0 && chosen[b] > key) {
                chosen[b + 1] = chosen[b];
                --b;
            }
            chosen[b + 1] = key;
        }
        float m = -INFINITY;
        for (int j = 0; j < p.k; ++j) m = fmaxf(m, lg[warp * p.E + chosen[j]]);
        float z = 0.f;
        for (int j = 0; j < p.k; ++j) z += expf(lg[warp * p.E + chosen[j]] - m);
        if (lane < p.k) {
            int e = chosen[0];
#pragma unroll
            for (int j = 1; j < kMaxTopK; ++j)
                if (j == lane) e = chosen[j];
            float w = expf(lg[warp * p.E + e] - m) / z;
            p.topk_idx[(size_t)t * p.k + lane] = e;
            p.topk_w[(size_t)t * p.k + lane] = w;
            __nv_bfloat16 wb = __float2bfloat16_rn(w);
            p.topk_wb[(size_t)t * p.k + lane] = *reinterpret_cast<uint16_t*>(&wb);
            atomicAdd(&p.hist[(size_t)(t / kChunkTokens) * p.E + e], 1);
        }
    }

    // ---- last CTA: histogram -> offsets, chunk bases, tile lists ----
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(p.done, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    __shared__ int s_count[kMaxExperts], s_off[kMaxExperts];
    for (int e = threadIdx.x; e < p.E; e += 256) {
        int run = 0;
        for (int c = 0; c < p.nchunks; ++c) run += __ldcg(&p.hist[(size_t)c * p.E + e]);
        s_count[e] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int off = 0, t1 = 0, t2 = 0;
        for (int e = 0; e < p.E; ++e) {
            int c = s_count[e];
            s_off[e] = off;
            p.offset[e] = off;
            p.count[e] = c;
            int mt = (c + 127) / 128;
            p.tiles1[e] = t1;
            p.tiles2[e] = t2;
            off += c;
            t1 += mt * p.nt1;
            t2 += mt * p.nt2;
        }
        p.offset[p.E] = off;
        p.tiles1[p.E] = t1;
        p.tiles2[p.E] = t2;
        p.status[kStatusTiles1] = (uint32_t)t1;
        p.status[kStatusTiles2] = (uint32_t)t2;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += 256) {
        int run = s_off[e];
        for (int c = 0; c < p.nchunks; ++c) {
            p.chunk_base[(size_t)c * p.E + e] = run;
            run += __ldcg(&p.hist[(size_t)c * p.E + e]);
        }
    }
}

cudaError_t launch_router(const RouteParams& p, cudaStream_t st) {
    const int Hx = (p.H + 7) & ~7;
    if (p.T <= 1024) {
        size_t sm = (size_t)Hx * 2 + (size_t)p.E * 4;
        cudaFuncSetAttribute(router_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        router_kernel<1><<<p.T, 256, sm, st>>>(p);
    } else {
        size_t sm = (size_t)4 * Hx * 2 + (size_t)4 * p.E * 4;
        cudaFuncSetAttribute(router_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        router_kernel<4><<<(p.T + 3) / 4, 256, sm, st>>>(p);
    }
    return cudaGetLastError();
}

// ======================================================= permute + x quant
// CTA = 8 warps over `tokens_per_cta` consecutive tokens (all in one 256-token
// chunk).  Row of (t, j) = chunk_base[chunk, e] + number of earlier tokens of
// the chunk routed to e, so rows are sorted by (expert, token).  Then each
// (token, 128-group) item is quantised by one warp: amax, s = amax/448,
// code = e4m3(x/s), written to each of the token's k rows.
__global__ void __launch_bounds__(256) permute_quant_kernel(PermuteParams p) {
    __shared__ int s_pre[kMaxExperts];
    __shared__ int s_idx[8 * kMaxTopK];
    __shared__ int s_row[8 * kMaxTopK];
    const int tpc = p.tokens_per_cta;
    const int t0 = blockIdx.x * tpc;
    const int chunk = t0 / kChunkTokens;
    const int c0 = chunk * kChunkTokens;
    const int nt = min(tpc, p.T - t0);
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) s_pre[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < (t0 - c0) * p.k; i += blockDim.x) atomicAdd(&s_pre[p.topk_idx[(size_t)c0 * p.k + i]], 1);
    for (int i = threadIdx.x; i < nt * p.k; i += blockDim.x) s_idx[i] = p.topk_idx[(size_t)t0 * p.k + i];
    __syncthreads();
    for (int i = threadIdx.x; i < nt * p.k; i += blockDim.x) {
        int tt = i / p.k, j = i - tt * p.k, e = s_idx[i];
        int r = p.chunk_base[(size_t)chunk * p.E + e] + s_pre[e];
        for (int u = 0; u < tt; ++u)
            for (int jj = 0; jj < p.k; ++jj) r += (s_idx[u * p.k + jj] == e);
        s_row[i] = r;
        int slot = (t0 + tt) * p.k + j;
        p.perm[r] = slot;
        p.inv[slot] = r;
    }
    __syncthreads();

    const int G = p.Hp / 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool vec = (p.H & 3) == 0;
    for (int item = warp; item < nt * G; item += 8) {
        const int tt = item / G, g = item - tt * G;
        const int t = t0 + tt;
        const int c = g * 128 + lane * 4;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        const uint16_t* xr = p.x + (size_t)t * p.H;
        if (vec && c + 4 <= p.H) {
            uint2 v = __ldg(reinterpret_cast<const uint2*>(xr + c));
            a[0] = __uint_as_float(v.x << 16);
            a[1] = __uint_as_float(v.x & 0xffff0000u);
            a[2] = __uint_as_float(v.y << 16);
            a[3] = __uint_as_float(v.y & 0xffff0000u);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = (c + i < p.H) ? bf16_bits_to_f32(xr[c + i]) : 0.f;
        }
        float amax = fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = group_scale(amax);
        const uint32_t q = quant4(a[0], a[1], a[2], a[3], s);
        for (int j = 0; j < p.k; ++j) {
            const int r = s_row[tt * p.k + j];
            *reinterpret_cast<uint32_t*>(p.xq + (size_t)r * p.Hp + c) = q;
            if (lane == 0) p.sx[(size_t)r * G + g] = s;
        }
    }
}

cudaError_t launch_permute_quant(const PermuteParams& p, cudaStream_t st) {
    int grid = (p.T + p.tokens_per_cta - 1) / p.tokens_per_cta;
    permute_quant_kernel<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

// ================================================================= combine
// out[t, n] = bf16_rn( sum_{j=0..k-1} part[t*k+j, n] ), slot order, fp32.
// ("Combine performs the weighted accumulation"; the weights were applied
// in the down GEMM's epilogue.)
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part, int T, int H, int ldp, int k,
                                                      uint16_t* __restrict__ out) {
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
    combine_kernel<<<grid, 256, 0, st>>>(part, T, H, ldp, k, out);
    return cudaGetLastError();
}

// ============================================================ weight packer
// One CTA per (128x128 destination block, expert).  Destination row dr maps
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
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) packed[i] = quant4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], sc);
    uint4* dst = reinterpret_cast<uint4*>(q + ((size_t)e * rows_p + dr) * cols_p + c0);
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
        *reinterpret_cast<uint32_t*>(q + (size_t)r * cp + c) = quant4(a[0], a[1], a[2], a[3], sc);
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
