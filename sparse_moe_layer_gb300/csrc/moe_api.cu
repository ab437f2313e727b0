// C ABI of the sparse MoE layer: argument checks, workspace carving, TMA
// tensor maps and the launch sequence
//   router -> permute + x quant -> gate/up GEMM -> down GEMM -> combine
// all on the caller's stream, with no allocation and no synchronisation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/moe_gb300.h"
#include "moe_device.cuh"
#include "moe_internal.h"

using namespace moe;

namespace {

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int pad128(int v) { return (v + 127) / 128 * 128; }

bool sizes_ok(int T, int H, int I, int E, int k) {
    if (T < 1 || H < 1 || I < 1 || E < 1 || k < 1) return false;
    if (E > kMaxExperts || k > kMaxTopK || k > E) return false;
    if (H > 16384 || I > 16384) return false;
    if ((long long)T * k >= (1LL << 31)) return false;
    return true;
}

// Decode-sized batches (few rows per expert) take the weight-streaming
// kernels with 32-row token tiles; larger ones the 128-row tile kernels.
inline bool decode_sized(long long R, int E) { return R <= 64LL * E; }


void layout_of(int T, int H, int I, int E, int k, moe_workspace_layout* L, bool mx = false) {
    const size_t R = (size_t)T * k;
    const size_t Hp = pad128(H), Ip = pad128(I);
    const size_t nch = (T + kChunkTokens - 1) / kChunkTokens;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->status = take(kStatusWords * 4);
    L->hist = take((nch * E + 1) * 4);  // + arrival counter of the router CTAs
    L->count = take((size_t)E * 4);
    L->offset = take((size_t)(E + 1) * 4);
    L->chunk_base = take(nch * E * 4);
    L->tiles1 = take((size_t)(E + 1) * 4);
    L->tiles2 = take((size_t)(E + 1) * 4);
    L->topk_idx = take(R * 4);
    L->topk_w = take(R * 4);
    L->topk_wb = take(R * 2);
    L->perm = take(R * 4);
    L->inv = take(R * 4);
    // MXFP8: scale atoms per (m-tile, K block); sum_e ceil(count_e/bm) <= E + ceil(R/bm) m-tiles
    const size_t bm = decode_sized((long long)R, E) ? 32 : 128;
    const size_t mt_bound = (size_t)E + (R + bm - 1) / bm;
    L->xq = take(R * Hp);
    L->sx = take(mx ? mt_bound * (Hp / 128) * kMxAtomBytes : R * (Hp / 128) * 4);
    L->hq = take(R * Ip);
    L->sh = take(mx ? mt_bound * (Ip / 128) * kMxAtomBytes : R * (Ip / 128) * 4);
    L->part = take(R * Hp * 4);
    L->total_bytes = o;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// 2D uint8 tensor [rows, cols] (row stride = cols bytes), box 128 bytes x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows = 128) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Blocked MXFP4 weight codes as a 2D tensor of 4-bit values [rows, 128], two
// per byte (64-byte rows), box 128 values x 128 rows, 128-byte swizzle.  The
// 16U4_ALIGN16B type lands each 16-value chunk in 16 bytes of shared memory
// (8 bytes of codes, 8 bytes of gap): the padded form the f8f6f4 MMA kinds
// read.  The type needs a 32-byte aligned base.
bool make_map_fp4(CUtensorMap* m, const void* base, uint64_t rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2D bf16 tensor [rows, cols] (row stride cols * 2 bytes, a multiple of 16),
// box 64 values (128 bytes) x box_rows, 128-byte swizzle; rows of the box past
// the tensor read as zeros.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Weight formats of forward_impl.
enum WeightFormat { kBlock128 = 0, kMxfp8 = 1, kMxfp4 = 2 };

}  // namespace

// What the router and the permutation kernel write (device pointers).
struct RoutingBuffers {
    uint32_t* status;     // uint32[64]; it and the zero_bytes after it are zeroed here
    size_t zero_bytes;    // the status words, the histogram and any counters placed after them
    int32_t* hist;        // [ceil(T/256), E] + 1 arrival counter (inside the zeroed bytes)
    int32_t* count;       // [E]
    int32_t* offset;      // [E+1]
    int32_t* chunk_base;  // [ceil(T/256), E]
    int32_t* tiles1;      // [E+1]
    int32_t* tiles2;      // [E+1]
    int32_t* topk_idx;    // [T, k]
    float* topk_w;        // [T, k]
    uint16_t* topk_wb;    // [T, k]
    int32_t* perm;        // [R]
    int32_t* inv;         // [R]
    uint8_t* xq;          // [R, Hp]
    float* sx;            // [Hp/128, R] (MXFP8: scale atoms)
};

// Steps a1-a4 on `st`: the status words and the histogram cleared, the router
// (top-k, softmax, per-chunk expert histogram), then the permutation with the
// x quantisation (1x128, or 1x32 MX when mx).  bm, nt1, nt2 size the GEMM tile
// lists the scan writes.  `mid` (optional) is recorded between the two kernels.
static moe_status launch_routing(const void* x, const void* router_w, const void* router_b, int T, int H, int E,
                                 int top_k, int bm, int nt1, int nt2, bool mx, const RoutingBuffers& b,
                                 cudaStream_t st, cudaEvent_t mid) {
    const int Hp = pad128(H);
    const int nch = (T + kChunkTokens - 1) / kChunkTokens;
    // status words, the (chunk, expert) histogram with its arrival counter, and
    // the counters after it start at zero
    if (cudaMemsetAsync(b.status, 0, b.zero_bytes, st) != cudaSuccess) return MOE_ERR_CUDA;
    RouteParams rp;
    rp.x = static_cast<const uint16_t*>(x);
    rp.rw = static_cast<const uint16_t*>(router_w);
    rp.rb = static_cast<const uint16_t*>(router_b);
    rp.T = T;
    rp.H = H;
    rp.E = E;
    rp.k = top_k;
    rp.nchunks = nch;
    rp.bm = bm;
    rp.nt1 = nt1;
    rp.nt2 = nt2;
    rp.topk_idx = b.topk_idx;
    rp.topk_w = b.topk_w;
    rp.topk_wb = b.topk_wb;
    rp.hist = b.hist;
    rp.done = b.hist + (size_t)nch * E;
    rp.count = b.count;
    rp.offset = b.offset;
    rp.chunk_base = b.chunk_base;
    rp.tiles1 = b.tiles1;
    rp.tiles2 = b.tiles2;
    rp.status = b.status;
    // large batches with 16-byte aligned rows: the tensor-core router
    if (const int np = router_tc_experts(T, H, E)) {
        CUtensorMap tmX, tmW;
        if (!make_map_bf16(&tmX, x, T, H, 128) || !make_map_bf16(&tmW, router_w, E, H, (uint32_t)np))
            return MOE_ERR_CUDA;
        if (launch_router_tc(rp, tmX, tmW, st) != cudaSuccess) return MOE_ERR_CUDA;
    } else if (launch_router(rp, st) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    if (mid) cudaEventRecord(mid, st);

    PermuteParams pp;
    pp.x = rp.x;
    pp.T = T;
    pp.H = H;
    pp.Hp = Hp;
    pp.E = E;
    pp.k = top_k;
    // 8 tokens per CTA for large batches while their x rows fit in 96 KB of shared memory
    pp.tokens_per_cta = (T > 2048 && 8LL * ((H + 7) & ~7) * 2 <= 96 * 1024) ? 8 : 1;
    pp.topk_idx = b.topk_idx;
    pp.chunk_base = b.chunk_base;
    pp.bm = bm;
    pp.nt1 = nt1;
    pp.offset = b.offset;
    pp.tiles1 = b.tiles1;
    pp.perm = b.perm;
    pp.inv = b.inv;
    pp.xq = b.xq;
    pp.R = T * top_k;
    pp.sx = b.sx;
    pp.mx = mx ? 1 : 0;
    pp.sxa = reinterpret_cast<uint8_t*>(b.sx);
    if (launch_permute_quant(pp, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

// How many n-tiles of each m-tile the decode down GEMM gives two w2 row
// blocks (j and j + P, j < P); the other RB - 2P take one, listed after all
// the paired tiles.  Two blocks per K step stream faster per byte than one
// (per K block ~0.75 us against ~0.48 us for one with 128x128 block scales),
// so every block that can be paired is, unless one-block tiles for the
// `active` experts that can have rows would not even fill the SMs.  (Fewer
// pairs, to even out the tiles per CTA, measured slower: one-block tiles in
// the paired kernel are no cheaper per byte.)
static int decode_down_pairs(int RB, int active, int sms) {
    return (long long)active * RB > sms ? RB / 2 : 0;
}

// Launch sequence shared by moe_forward and moe_forward_profiled; when `ev`
// is non-null, ev[i] is recorded on the stream before stage i and ev[5]
// after the last stage.
// fmt: kBlock128 (e4m3 codes, fp32 128x128 block scales), kMxfp8 (e4m3 codes,
// UE8M0 scale atoms) or kMxfp4 (E2M1 codes two per byte, UE8M0 scale atoms).
static moe_status forward_impl(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                               const void* s13, const void* b13, const uint8_t* w2, const void* s2, const void* b2,
                               int T, int H, int I, int E, int top_k, void* out, void* workspace,
                               size_t workspace_bytes, void* stream, void* const* ev, int fmt = kBlock128);

extern "C" {

size_t moe_workspace_size(int T, int H, int I, int E, int top_k) {
    if (!sizes_ok(T, H, I, E, top_k)) return 0;
    moe_workspace_layout L;
    layout_of(T, H, I, E, top_k, &L);
    return L.total_bytes;
}

moe_status moe_get_workspace_layout(int T, int H, int I, int E, int top_k, moe_workspace_layout* layout) {
    if (!layout || !sizes_ok(T, H, I, E, top_k)) return MOE_ERR_INVALID_ARG;
    layout_of(T, H, I, E, top_k, layout);
    return MOE_OK;
}

moe_status moe_forward(const void* x, const void* router_w, const void* router_b, const uint8_t* w13, const float* s13,
                       const void* b13, const uint8_t* w2, const float* s2, const void* b2, int T, int H, int I, int E,
                       int top_k, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, nullptr);
}

moe_status moe_forward_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                const float* s13, const void* b13, const uint8_t* w2, const float* s2, const void* b2,
                                int T, int H, int I, int E, int top_k, void* out, void* workspace,
                                size_t workspace_bytes, void* stream, void* const* events) {
    if (!events) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, events);
}

size_t moe_workspace_size_mx(int T, int H, int I, int E, int top_k) {
    if (!sizes_ok(T, H, I, E, top_k)) return 0;
    moe_workspace_layout L;
    layout_of(T, H, I, E, top_k, &L, true);
    return L.total_bytes;
}

moe_status moe_get_workspace_layout_mx(int T, int H, int I, int E, int top_k, moe_workspace_layout* layout) {
    if (!layout || !sizes_ok(T, H, I, E, top_k)) return MOE_ERR_INVALID_ARG;
    layout_of(T, H, I, E, top_k, layout, true);
    return MOE_OK;
}

moe_status moe_forward_mx(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                          const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2, const void* b2,
                          int T, int H, int I, int E, int top_k, void* out, void* workspace, size_t workspace_bytes,
                          void* stream) {
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, nullptr, kMxfp8);
}

moe_status moe_forward_mx_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                   const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2,
                                   const void* b2, int T, int H, int I, int E, int top_k, void* out, void* workspace,
                                   size_t workspace_bytes, void* stream, void* const* events) {
    if (!events) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, events, kMxfp8);
}

moe_status moe_forward_mxfp4(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                             const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2, const void* b2,
                             int T, int H, int I, int E, int top_k, void* out, void* workspace, size_t workspace_bytes,
                             void* stream) {
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, nullptr, kMxfp4);
}

moe_status moe_forward_mxfp4_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                      const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2,
                                      const void* b2, int T, int H, int I, int E, int top_k, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream, void* const* events) {
    if (!events) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, workspace,
                        workspace_bytes, stream, events, kMxfp4);
}

}  // extern "C"

static moe_status forward_impl(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                               const void* s13, const void* b13, const uint8_t* w2, const void* s2, const void* b2,
                               int T, int H, int I, int E, int top_k, void* out, void* workspace,
                               size_t workspace_bytes, void* stream, void* const* ev, int fmt) {
    const bool mx = fmt != kBlock128;
    auto mark = [&](int i) {
        if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), static_cast<cudaStream_t>(stream));
    };
    if (!x || !router_w || !router_b || !w13 || !s13 || !b13 || !w2 || !s2 || !b2 || !out || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!sizes_ok(T, H, I, E, top_k)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(w13) || !aligned16(w2) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_UNSUPPORTED;
    if (mx && (!aligned16(s13) || !aligned16(s2))) return MOE_ERR_UNSUPPORTED;  // scale atoms move by bulk copy
    if (fmt == kMxfp4 && (!aligned32(w13) || !aligned32(w2))) return MOE_ERR_UNSUPPORTED;  // 4-bit tensor maps
    moe_workspace_layout L;
    layout_of(T, H, I, E, top_k, &L, mx);
    if (workspace_bytes < L.total_bytes) return MOE_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int Hp = pad128(H), Ip = pad128(I);
    const int R = T * top_k;
    const int sms = num_sms();

    mark(0);

    // Few rows per expert (decode): weight-streaming kernels with 32-row token
    // tiles and 128-feature n-tiles; else 128-row tiles of 128 h features
    // (gate/up) or 256 output features (down: two w2 blocks per tile).
    const bool decode = decode_sized(R, E);
    const int bm = decode ? 32 : 128;
    const int nt1 = Ip / 128;
    // Decode down GEMM: the first `pairs` n-tiles of every m-tile take two w2
    // row blocks, the rest one (decode_down_pairs).
    const int pairs = decode ? decode_down_pairs(Hp / 128, E < R ? E : R, sms) : 0;
    const int nt2 = decode ? Hp / 128 - pairs : (Hp / 128 + 1) / 2;
    RoutingBuffers rb;
    rb.status = reinterpret_cast<uint32_t*>(ws + L.status);
    rb.zero_bytes = L.count - L.status;
    rb.hist = reinterpret_cast<int32_t*>(ws + L.hist);
    rb.count = reinterpret_cast<int32_t*>(ws + L.count);
    rb.offset = reinterpret_cast<int32_t*>(ws + L.offset);
    rb.chunk_base = reinterpret_cast<int32_t*>(ws + L.chunk_base);
    rb.tiles1 = reinterpret_cast<int32_t*>(ws + L.tiles1);
    rb.tiles2 = reinterpret_cast<int32_t*>(ws + L.tiles2);
    rb.topk_idx = reinterpret_cast<int32_t*>(ws + L.topk_idx);
    rb.topk_w = reinterpret_cast<float*>(ws + L.topk_w);
    rb.topk_wb = reinterpret_cast<uint16_t*>(ws + L.topk_wb);
    rb.perm = reinterpret_cast<int32_t*>(ws + L.perm);
    rb.inv = reinterpret_cast<int32_t*>(ws + L.inv);
    rb.xq = ws + L.xq;
    rb.sx = reinterpret_cast<float*>(ws + L.sx);
    {
        const moe_status rs = launch_routing(x, router_w, router_b, T, H, E, top_k, bm, nt1, nt2, mx, rb, st,
                                             ev ? static_cast<cudaEvent_t>(ev[1]) : nullptr);
        if (rs != MOE_OK) return rs;
    }
    mark(2);

    // upper bound of the tile count of either GEMM: sum_e ceil(count_e/bm) <= E + R/bm
    const long long mt_bound = (long long)E + (R + bm - 1) / bm;

    CUtensorMap tmA1, tmB1, tmA2, tmB2;
    // weights are blocked: a 2D view of 128-byte rows, one 128x128 block = 128 consecutive rows
    // decode kernels load a tile's activation rows in boxes of kDecXBoxRows, only as many as it has rows
    const uint32_t a_box = decode ? kDecXBoxRows : (uint32_t)bm;
    const uint64_t rows13 = (uint64_t)E * 2 * Ip * (Hp / 128), rows2 = (uint64_t)E * Hp * (Ip / 128);
    const bool wmaps = fmt == kMxfp4 ? make_map_fp4(&tmB1, w13, rows13) && make_map_fp4(&tmB2, w2, rows2)
                                     : make_map(&tmB1, w13, rows13, 128) && make_map(&tmB2, w2, rows2, 128);
    if (!wmaps || !make_map(&tmA1, rb.xq, R, Hp, a_box) || !make_map(&tmA2, ws + L.hq, R, Ip, a_box))
        return MOE_ERR_CUDA;

    if (mx) {
        MxGemmParams m1;
        memset(&m1, 0, sizeof(m1));
        m1.E = E;
        m1.R = R;
        m1.KB = Hp / 128;
        m1.N_real = I;
        m1.sw_rowblocks = 2 * Ip / 128;
        m1.up_rows = Ip;
        m1.nt = nt1;
        m1.count = rb.count;
        m1.offset = rb.offset;
        m1.tiles = rb.tiles1;
        m1.sa = ws + L.sx;
        m1.sw = static_cast<const uint8_t*>(s13);
        m1.bias = static_cast<const uint16_t*>(b13);
        m1.hq = ws + L.hq;
        m1.sh = ws + L.sh;
        m1.ldq = Ip;
        m1.status = rb.status;
        const long long t1 = mt_bound * nt1;
        if (launch_gemm_mx(true, decode, fmt == kMxfp4, tmA1, tmB1, m1, (int)(t1 < sms ? t1 : sms), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(3);
        MxGemmParams m2;
        memset(&m2, 0, sizeof(m2));
        m2.E = E;
        m2.R = R;
        m2.KB = Ip / 128;
        m2.N_real = H;
        m2.sw_rowblocks = Hp / 128;
        m2.up_rows = pairs * 128;  // paired tile j < pairs: w2 row blocks j and j + pairs
        m2.nt = nt2;
        m2.count = rb.count;
        m2.offset = rb.offset;
        m2.tiles = rb.tiles2;
        m2.sa = ws + L.sh;
        m2.sw = static_cast<const uint8_t*>(s2);
        m2.bias = static_cast<const uint16_t*>(b2);
        m2.perm = rb.perm;
        m2.topk_wb = rb.topk_wb;
        m2.part = reinterpret_cast<float*>(ws + L.part);
        m2.ldp = Hp;
        m2.status = rb.status;
        const long long t2 = mt_bound * nt2;
        if (launch_gemm_mx(false, decode, fmt == kMxfp4, tmA2, tmB2, m2, (int)(t2 < sms ? t2 : sms), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(4);
        if (launch_combine(m2.part, T, H, Hp, top_k, static_cast<uint16_t*>(out), sms, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(5);
        return MOE_OK;
    }

    GemmParams g1;
    memset(&g1, 0, sizeof(g1));
    g1.E = E;
    g1.R = R;
    g1.KB = Hp / 128;
    g1.N_real = I;
    g1.rows_B = 2 * Ip;
    g1.up_rows = Ip;
    g1.sw_rowblocks = 2 * Ip / 128;
    g1.count = rb.count;
    g1.offset = rb.offset;
    g1.tiles = rb.tiles1;
    g1.sa = rb.sx;
    g1.sw = static_cast<const float*>(s13);
    g1.bias = static_cast<const uint16_t*>(b13);
    g1.hq = ws + L.hq;
    g1.sh = reinterpret_cast<float*>(ws + L.sh);
    g1.ldq = Ip;
    g1.status = rb.status;
    long long t1 = mt_bound * (Ip / 128);
    int grid1 = (int)(t1 < sms ? t1 : sms);
    if ((decode ? launch_gemm_gateup_decode(tmB1, tmA1, g1, grid1, st) : launch_gemm_gateup(tmA1, tmB1, g1, grid1, st))
        != cudaSuccess)
        return MOE_ERR_CUDA;
    mark(3);

    GemmParams g2;
    memset(&g2, 0, sizeof(g2));
    g2.E = E;
    g2.R = R;
    g2.KB = Ip / 128;
    g2.N_real = H;
    g2.rows_B = Hp;
    g2.up_rows = pairs * 128;  // paired tile j < pairs: w2 row blocks j and j + pairs
    g2.sw_rowblocks = Hp / 128;
    g2.count = rb.count;
    g2.offset = rb.offset;
    g2.tiles = rb.tiles2;
    g2.sa = g1.sh;
    g2.sw = static_cast<const float*>(s2);
    g2.bias = static_cast<const uint16_t*>(b2);
    g2.perm = rb.perm;
    g2.topk_wb = rb.topk_wb;
    g2.part = reinterpret_cast<float*>(ws + L.part);
    g2.ldp = Hp;
    g2.status = rb.status;
    long long t2 = mt_bound * nt2;
    int grid2 = (int)(t2 < sms ? t2 : sms);
    if ((decode ? launch_gemm_down_decode(tmB2, tmA2, g2, grid2, st) : launch_gemm_down(tmA2, tmB2, g2, grid2, st)) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    mark(4);

    if (launch_combine(g2.part, T, H, Hp, top_k, static_cast<uint16_t*>(out), sms, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    mark(5);
    return MOE_OK;
}

// ---------------------------------------------------------------------------
// Forward with a library-owned scratch area, for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc: plugins whose device memory belongs to
// a host framework's caching allocator or a serving engine's fixed memory
// pool, and code that must keep cudaMalloc/cudaFree (and the synchronisation
// cudaFree implies) out of its latency path.  For them the layer's scratch
// lives in this file-scope device array: every GPU that loads the library
// holds it until the process exits, and every call on a device shares it.
// Host code must not pass g_static_scratch itself to a kernel -- in host code
// that name is a host-side stand-in, not a device address -- so the device
// address is looked up once per device with cudaGetSymbolAddress.
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;  // 32 MiB
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// Per device: the context the address was looked up in, and the address.  A
// context torn down and made again (cudaDeviceReset, or the primary context
// released and retained anew) loads the module again, possibly elsewhere, so
// the address is looked up again whenever the current context differs.
struct ScratchAddr {
    CUcontext ctx;
    void* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

CUcontext current_context() {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    });
    CUcontext c = nullptr;
    if (!g_ctx_current || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of g_static_scratch on the current device, looked up with
// cudaGetSymbolAddress the first time in each context (that first lookup may
// load the module, so it must not happen inside a stream capture).
moe_status static_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& a = g_scratch_addr[dev];
    const CUcontext now = current_context();
    if (!a.ptr || !now || a.ctx != now) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        a.ptr = p;
        a.ctx = current_context();  // the lookup above made the context current if none was
    }
    *out = a.ptr;
    return MOE_OK;
}
}  // namespace

extern "C" moe_status moe_forward_static_scratch(const void* x, const void* router_w, const void* router_b,
                                                 const uint8_t* w13, const float* s13, const void* b13,
                                                 const uint8_t* w2, const float* s2, const void* b2, int T, int H,
                                                 int I, int E, int top_k, void* out, void* stream) {
    // argument errors first, then the size limit of the static array
    if (!x || !router_w || !router_b || !w13 || !s13 || !b13 || !w2 || !s2 || !b2 || !out) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_workspace_size(T, H, I, E, top_k);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // these sizes need more than the static area
    void* scratch = nullptr;
    const moe_status st = static_scratch_address(&scratch);
    if (st != MOE_OK) return st;
    // forward_impl clears the status words and the expert histogram at the
    // start of every call, so nothing left by the previous call leaks in.
    return forward_impl(x, router_w, router_b, w13, s13, b13, w2, s2, b2, T, H, I, E, top_k, out, scratch,
                        kStaticScratchBytes, stream, nullptr);
}

// The device error word of the static array (its first word, as in a
// caller's workspace): read after synchronising the stream, then cleared.
extern "C" moe_status moe_read_static_scratch_status(void* stream) {
    void* scratch = nullptr;
    const moe_status st = static_scratch_address(&scratch);
    if (st != MOE_OK) return st;
    return moe_read_device_status(scratch, stream);
}

// Workspace of moe_route_debug: the intermediates of the routing steps that
// the caller does not ask for, carved like the forward's workspace.
namespace {
struct RouteLayout {
    size_t status, hist, count, chunk_base, tiles1, tiles2, topk_wb, inv, total;
};
RouteLayout route_layout_of(int T, int E, int k) {
    const size_t R = (size_t)T * k;
    const size_t nch = (T + kChunkTokens - 1) / kChunkTokens;
    RouteLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.status = take(kStatusWords * 4);
    L.hist = take((nch * E + 1) * 4);
    L.count = take((size_t)E * 4);
    L.chunk_base = take(nch * E * 4);
    L.tiles1 = take((size_t)(E + 1) * 4);
    L.tiles2 = take((size_t)(E + 1) * 4);
    L.topk_wb = take(R * 2);
    L.inv = take(R * 4);
    L.total = o;
    return L;
}
}  // namespace

extern "C" size_t moe_route_workspace_size(int T, int H, int E, int top_k) {
    if (!sizes_ok(T, H, 1, E, top_k)) return 0;
    return route_layout_of(T, E, top_k).total;
}

extern "C" moe_status moe_route_debug(const void* x, const void* router_w, const void* router_b, int T, int H, int E,
                                      int top_k, int32_t* topk_idx, float* topk_w, int32_t* offset, int32_t* perm,
                                      uint8_t* xq, float* sx, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    if (!x || !router_w || !router_b || !topk_idx || !topk_w || !offset || !perm || !xq || !sx || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!sizes_ok(T, H, 1, E, top_k)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(xq) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_UNSUPPORTED;
    const RouteLayout L = route_layout_of(T, E, top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    RoutingBuffers b;
    b.status = reinterpret_cast<uint32_t*>(ws + L.status);
    b.zero_bytes = L.count - L.status;
    b.hist = reinterpret_cast<int32_t*>(ws + L.hist);
    b.count = reinterpret_cast<int32_t*>(ws + L.count);
    b.offset = offset;
    b.chunk_base = reinterpret_cast<int32_t*>(ws + L.chunk_base);
    b.tiles1 = reinterpret_cast<int32_t*>(ws + L.tiles1);
    b.tiles2 = reinterpret_cast<int32_t*>(ws + L.tiles2);
    b.topk_idx = topk_idx;
    b.topk_w = topk_w;
    b.topk_wb = reinterpret_cast<uint16_t*>(ws + L.topk_wb);
    b.perm = perm;
    b.inv = reinterpret_cast<int32_t*>(ws + L.inv);
    b.xq = xq;
    b.sx = sx;
    // the GEMM tile lists are not asked for: one n-tile per m-tile of the forward's row tiling
    const int bm = decode_sized((long long)T * top_k, E) ? 32 : 128;
    return launch_routing(x, router_w, router_b, T, H, E, top_k, bm, 1, 1, false, b,
                          static_cast<cudaStream_t>(stream), nullptr);
}

extern "C" moe_status moe_block_weights(const uint8_t* w13_rm, const uint8_t* w2_rm, int H, int I, int E,
                                        uint8_t* w13, uint8_t* w2, void* stream) {
    if (H < 1 || I < 1 || E < 1 || H > 16384 || I > 16384 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (!w13_rm && !w2_rm) return MOE_ERR_INVALID_ARG;
    if ((w13_rm && !w13) || (w2_rm && !w2)) return MOE_ERR_INVALID_ARG;
    if ((w13_rm && (!aligned16(w13_rm) || !aligned16(w13))) || (w2_rm && (!aligned16(w2_rm) || !aligned16(w2))))
        return MOE_ERR_UNSUPPORTED;
    const int Hp = pad128(H), Ip = pad128(I);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (w13_rm && launch_block_codes(w13_rm, E, 2 * Ip, Hp, w13, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (w2_rm && launch_block_codes(w2_rm, E, Hp, Ip, w2, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

extern "C" {

moe_status moe_pack_weights(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13, float* s13,
                            uint8_t* w2, float* s2, void* stream) {
    if (H < 1 || I < 1 || E < 1 || H > 16384 || I > 16384 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (!w13_f32 && !w2_f32) return MOE_ERR_INVALID_ARG;
    if ((w13_f32 && (!w13 || !s13)) || (w2_f32 && (!w2 || !s2))) return MOE_ERR_INVALID_ARG;
    if ((w13 && !aligned16(w13)) || (w2 && !aligned16(w2))) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Hp = pad128(H), Ip = pad128(I);
    if (w13_f32 && launch_pack_blocks(w13_f32, E, 2 * I, H, 2 * Ip, Hp, I, w13, s13, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (w2_f32 && launch_pack_blocks(w2_f32, E, H, I, Hp, Ip, 0, w2, s2, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_pack_weights_mx(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13,
                               uint8_t* s13, uint8_t* w2, uint8_t* s2, void* stream) {
    if (H < 1 || I < 1 || E < 1 || H > 16384 || I > 16384 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (!w13_f32 && !w2_f32) return MOE_ERR_INVALID_ARG;
    if ((w13_f32 && (!w13 || !s13)) || (w2_f32 && (!w2 || !s2))) return MOE_ERR_INVALID_ARG;
    if ((w13 && !aligned16(w13)) || (w2 && !aligned16(w2)) || (s13 && !aligned16(s13)) || (s2 && !aligned16(s2)))
        return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Hp = pad128(H), Ip = pad128(I);
    if (w13_f32 && launch_pack_blocks_mx(w13_f32, E, 2 * I, H, 2 * Ip, Hp, I, w13, s13, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (w2_f32 && launch_pack_blocks_mx(w2_f32, E, H, I, Hp, Ip, 0, w2, s2, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_pack_weights_mxfp4(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13,
                                  uint8_t* s13, uint8_t* w2, uint8_t* s2, void* stream) {
    if (H < 1 || I < 1 || E < 1 || H > 16384 || I > 16384 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (!w13_f32 && !w2_f32) return MOE_ERR_INVALID_ARG;
    if ((w13_f32 && (!w13 || !s13)) || (w2_f32 && (!w2 || !s2))) return MOE_ERR_INVALID_ARG;
    if ((w13 && !aligned16(w13)) || (w2 && !aligned16(w2)) || (s13 && !aligned16(s13)) || (s2 && !aligned16(s2)))
        return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int Hp = pad128(H), Ip = pad128(I);
    if (w13_f32 && launch_pack_blocks_mx4(w13_f32, E, 2 * I, H, 2 * Ip, Hp, I, w13, s13, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (w2_f32 && launch_pack_blocks_mx4(w2_f32, E, H, I, Hp, Ip, 0, w2, s2, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_quantize_rows_mx(const float* in, int rows, int cols, int ld_in, uint8_t* q, uint8_t* s,
                                void* stream) {
    if (!in || !q || !s || rows < 1 || cols < 1 || ld_in < cols) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 3u) return MOE_ERR_UNSUPPORTED;
    if (launch_quantize_rows_mx(in, rows, cols, ld_in, q, s, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_quantize_rows(const float* in, int rows, int cols, int ld_in, uint8_t* q, float* s, void* stream) {
    if (!in || !q || !s || rows < 1 || cols < 1 || ld_in < cols) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 3u) return MOE_ERR_UNSUPPORTED;
    if (launch_quantize_rows(in, rows, cols, ld_in, q, s, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_read_device_status(void* workspace, void* stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(workspace, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
    return word ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

moe_status moe_test_bounded_wait(uint64_t timeout_ns, int arrivals, uint32_t* result_dev, void* stream) {
    if (!result_dev || arrivals < 0 || arrivals > 1) return MOE_ERR_INVALID_ARG;
    if (launch_bounded_wait_test(timeout_ns, arrivals, result_dev, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported (alignment or size limit)";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA launch or runtime error";
        case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
