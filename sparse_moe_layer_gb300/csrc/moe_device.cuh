// Device helpers shared by the layer's kernels: bf16/e4m3 conversion, the 1x128
// group quantiser, and thin inline-PTX wrappers for mbarrier, TMA and tcgen05
// (sm_103a).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- limits ----
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 256;
constexpr int kChunkTokens = 256;  // token chunk of the expert histogram
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // every device wait gives up after 2 s

// status words (uint32 array at the head of the workspace)
enum : int {
    kStatusError = 0,
    kStatusTiles1 = 1,
    kStatusTiles2 = 2,
    kStatusTileRows = 3,
    kStatusWords = 64
};
enum : uint32_t { kErrTimeoutProducer = 1u, kErrTimeoutMma = 2u, kErrTimeoutEpilogue = 4u };

// ------------------------------------------------------------ conversion ----
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 -> two e4m3 codes, round to nearest even, saturating to +-448.
// Returns lo_val's code in bits [0,8) and hi_val's in bits [8,16).
__device__ __forceinline__ uint32_t e4m3x2(float lo_val, float hi_val) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi_val), "f"(lo_val));
    return (uint32_t)r;
}

// Scale of one 128-wide group from its absolute maximum: amax/448 in IEEE
// fp32, 1 for an all-zero group (its codes are then all +0).
__device__ __forceinline__ float group_scale(float amax) { return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f); }

// The correctly rounded fp32 quotient v/s, given r = RN(1/s): q0 = RN(v*r),
// rem = v - q0*s (exact with one FMA), q = RN(q0 + rem*r) -- Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 1990).  The remainder is
// exact while it stays in the normal range, which holds for |v| >= 2^-96
// (then s >= |v|/448 is normal as well).  The quantisers divide every value
// of a 1x128 group by the group's scale s = amax/448, and when amax >= 2^-64
// the values below 2^-96 have |v/s| < 448*2^-32, far below half the smallest
// e4m3 subnormal (2^-10): their code is the signed zero whatever the step
// returns, as long as the sign is v's.  So div_fast ends by setting the sign
// bit from v (keep = sign_keep(amax)), which also keeps the sign of -0; in an
// all-zero group (amax = 0, s = 1) it clears the sign instead, so that every
// code of that group is +0.  Groups with 0 < amax < 2^-64 take IEEE division
// (quot_fast false).  Either way the e4m3 codes are those of the correctly
// rounded quotient, bit for bit (checked by the quantiser tests, tiny,
// all-zero and signed-zero groups included).
__device__ __forceinline__ float recip_rn(float s) { return __frcp_rn(s); }
__device__ __forceinline__ bool quot_fast(float amax) { return !(amax > 0.0f && amax < 0x1p-64f); }
__device__ __forceinline__ uint32_t sign_keep(float amax) { return amax == 0.0f ? 0u : 0x80000000u; }
__device__ __forceinline__ float div_fast(float v, float s, float r, uint32_t keep) {
    const float q0 = __fmul_rn(v, r);
    const float rem = __fmaf_rn(-q0, s, v);
    const float q = __fmaf_rn(rem, r, q0);
    return __uint_as_float((__float_as_uint(q) & 0x7fffffffu) | (__float_as_uint(v) & keep));
}

// Four values of a group with absolute maximum amax, scale s = group_scale(amax)
// and r = recip_rn(s) -> four e4m3 codes (byte i = value i).
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float amax, float s, float r) {
    if (quot_fast(amax)) {
        const uint32_t k = sign_keep(amax);
        return e4m3x2(div_fast(a, s, r, k), div_fast(b, s, r, k)) |
               (e4m3x2(div_fast(c, s, r, k), div_fast(d, s, r, k)) << 16);
    }
    return e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s)) | (e4m3x2(__fdiv_rn(c, s), __fdiv_rn(d, s)) << 16);
}

// ----------------------------------------------------- MXFP8 quantiser ----
// OCP Microscaling Formats (MX) v1.0, section 6.3, for a group of 32 values
// with absolute maximum amax: shared exponent X = floor(log2(amax)) - 8 (8 =
// the exponent of e4m3's largest normal), stored as the UE8M0 byte X + 127;
// codes e4m3_rne_satfinite(v * 2^-X).  X is clamped to [-127, 127] and an
// all-zero group gets the byte 0 and +0 codes.  For amax > 0 with biased
// fp32 exponent b (0 for a subnormal amax), floor(log2(amax)) = b - 127 for
// a normal amax, and every amax below 2^-119 lands on the clamp, so the
// byte is max(b - 8, 0); a finite amax never reaches the upper clamp.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
    const int b = (int)((__float_as_uint(amax) >> 23) & 0xffu);
    return amax == 0.0f ? 0u : (uint32_t)max(b - 8, 0);
}
// 2^-X = 2^(127 - byte) as an fp32 (a normal number for every byte in [0, 246]).
__device__ __forceinline__ float mx_inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }
// Sign mask of a group's scaled values: an all-zero group's codes are +0.
__device__ __forceinline__ uint32_t mx_keep(float amax) { return amax == 0.0f ? 0x7fffffffu : 0xffffffffu; }
// v * 2^-X rounded once to fp32 (exact unless it underflows, and then far
// below the smallest e4m3 subnormal), sign-masked.
__device__ __forceinline__ float mx_scaled(float v, float inv, uint32_t keep) {
    return __uint_as_float(__float_as_uint(__fmul_rn(v, inv)) & keep);
}
__device__ __forceinline__ uint32_t mx_quant4(float a, float b, float c, float d, float inv, uint32_t keep) {
    return e4m3x2(mx_scaled(a, inv, keep), mx_scaled(b, inv, keep)) |
           (e4m3x2(mx_scaled(c, inv, keep), mx_scaled(d, inv, keep)) << 16);
}

// Scale atoms.  The block-scaled MMA (kind::mxf8f6f4, scale_vec::1X) reads
// the scale of A row m from TMEM lane m, column sfa + m/32, and the scale of
// B column n from the lane (n mod 32) of the accumulator row's lane quarter,
// column sfb + n/32; the byte of the 32-bit cell is the MMA's scale id, here
// the 32-wide K group inside a 128-wide K block.  tcgen05.cp 32x128b.warpx4
// copies 32 rows of 16 bytes into 4 columns of lanes 0-31 and replicates
// them into the other three quarters, so one 512-byte atom serves 128 rows
// (or columns) x one K block: byte (r % 32) * 16 + (r / 32) * 4 + g for row
// r and K group g.  Weight blocks, activation tiles and token tiles all use
// this atom.
__host__ __device__ constexpr int mx_atom_byte(int r, int g) { return (r & 31) * 16 + (r >> 5) * 4 + g; }
constexpr int kMxAtomBytes = 512;

// 2^x and 1/x from the special-function unit (PTX ex2.approx / rcp.approx,
// subnormals flushed): one instruction each, no branches.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// h[i] = silu(g[i]) * u[i] = g * u / (1 + e^-g) for i < N, written over g;
// h = 0 for i >= n_valid (padding features).  Returns max_i |h[i]|.
// e^-g = 2^(-g log2 e); both special-function operations are the hardware
// approximations (a few ulp, no branches), issued in independent batches of
// 16 so they overlap.
template <int N>
__device__ __forceinline__ float swiglu_inplace(float* g, const float* u, int n_valid) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int b = 0; b < N; b += 16) {
        float e[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) e[i] = ex2_approx(g[b + i] * kNegLog2e);
#pragma unroll
        for (int i = 0; i < 16; ++i) e[i] = rcp_approx(1.0f + e[i]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float h = (b + i < n_valid) ? g[b + i] * e[i] * u[b + i] : 0.f;
            g[b + i] = h;
            m[i & 3] = fmaxf(m[i & 3], fabsf(h));
        }
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Max over the 32 lanes of column j of v (each lane holds one row of 32
// values), returned in lane j: a transpose-and-reduce butterfly that halves
// the columns a lane keeps at every step (31 shuffles instead of 32 x 5).
// v is overwritten.
__device__ __forceinline__ float column_max32(float (&v)[32], int lane) {
#pragma unroll
    for (int n = 16; n >= 1; n >>= 1) {
        const bool hi = (lane & n) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = hi ? v[i] : v[i + n];
            const float keep = hi ? v[i + n] : v[i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, n));
        }
    }
    return v[0];
}

// ------------------------------------------------------------- smem/ptx ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false when the
// wait gave up (after timeout_ns) or when another role has already aborted
// (*abort != 0); on a timeout it raises *abort and ORs err_bit into *err.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t* err,
                                          uint32_t err_bit, uint64_t timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > timeout_ns) {
            *abort = 1;
            if (err) atomicOr(err, err_bit);
            return false;
        }
    }
}

// ------------------------------------------------------- thread-block cluster ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes made
// before it are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr(local_addr, rank)) : "memory");
    return v;
}
// ------------------------------------------------------------------ TMA ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2D tiled load of one box (inner coordinate x in elements, row y) into
// shared memory, completing transaction bytes on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// -------------------------------------------------------------- tcgen05 ----
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzled
// layout (rows of 128 bytes, 8-row atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);        // start address
    d |= (uint64_t)1 << 16;                       // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: 8 rows * 128 B
    d |= (uint64_t)1 << 46;                       // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = e4m3, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                       // D format fp32
           | (0u << 7) | (0u << 10)        // A, B format e4m3
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void mma_e4m3(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                       // D format fp32
           | (1u << 7) | (1u << 10)        // A, B format bf16
           | ((uint32_t)(N >> 3) << 17)    // N / 8
           | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D (+)= A * B^T with 16-bit operands (K = 16 per instruction).
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled MMA (kind::mxf8f6f4, one UE8M0 scale per 32 K values of each
// A row and each B column): instruction descriptor without the scale ids
// (A = B = e4m3, fp32 D, both K-major, bit 23 = UE8M0 scales) ...
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N) {
    return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
// Operand format codes of the f8f6f4 kinds (A: bits 7-9, B: bits 10-12):
// e4m3 = 0, e2m1 (FP4) = 5.  An e2m1 operand sits in shared memory in the
// padded form: each 16-byte chunk holds 16 packed 4-bit values in its first 8
// bytes, so a 128-value K block still spans one 128-byte row.
constexpr uint32_t kFmtE4M3 = 0, kFmtE2M1 = 5;
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t afmt, uint32_t bfmt) {
    return idesc_mx_e4m3(M, N) | (afmt << 7) | (bfmt << 10);
}
// ... with the byte of the scale cells this MMA reads (B: bits 4-5, A: bits 29-30).
__device__ __forceinline__ uint32_t idesc_sf_id(uint32_t idesc, uint32_t id) { return idesc | (id << 4) | (id << 29); }

__device__ __forceinline__ void mma_mx(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of one 512-byte scale atom (32 rows of 16 bytes,
// no swizzle: 8-row groups 128 bytes apart) ...
__device__ __forceinline__ uint64_t smem_desc_atom(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)(128 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}
// ... copied into TMEM columns [taddr, taddr + 4) of every lane quarter.
// Ordered before the MMAs this thread issues after it.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint32_t smem_addr) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(smem_desc_atom(smem_addr))
                 : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane, then the wait
// for them.  The wait names the registers as operands so that no use of them
// can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}


// 16 consecutive 32-bit columns of this thread's TMEM lane, then the wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel in the stream
// has completed and its writes are visible (returns at once when this grid
// was launched without the attribute) ...
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// ... and let the next kernel in the stream be scheduled once every CTA of
// this grid has executed this (or exited).
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }


// 64 consecutive 32-bit columns of this thread's TMEM lane (two x32 loads
// issued back to back), then one wait for both.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr), "r"(taddr + 32u));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
                 :
                 : "memory");
}

// Hand registers between warpgroups (all four warps of a warpgroup execute it).
template <int N>
__device__ __forceinline__ void regs_release() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_acquire() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace moe
