/*
 * moe_gb300 -- forward pass of a gpt-oss-style sparse Mixture-of-Experts MLP
 * layer on one GB300 (sm_103a).  Plain C ABI: device pointers, sizes, a
 * CUDA stream passed as void*.
 *
 * The layer (as stated in "GPT-OSS on Day 0", perplexity.ai hub blog: the MLP
 * bullets of the gpt-oss architecture list -- SwiGLU, softmax after top-k,
 * experts with biases; the infrastructure decisions -- FP8 with 128x128 block
 * scales; the MoE routing, DeepGEMM bias and combine paragraphs):
 *
 *   logits[t,e] = sum_h x[t,h] * router_w[e,h] + router_b[e]          (fp32)
 *   the k largest logits (ties -> lower e), stored in ascending expert order
 *   w[t,j]      = softmax over those k logits, rounded to bf16
 *   rows of each expert e (tokens routed to e, ascending token order):
 *     xq, sx    = 1x128 per-token-group FP8 e4m3 quantisation of x
 *                 (s = amax/448, code = e4m3_rne_satfinite(x/s))
 *     acc       = b13[e] + sum_kb sx[kb]*s13[e,n/128,kb] * (xq . w13[e,n])_kb
 *     h         = silu(gate) * up,  requantised 1x128 -> hq, sh
 *     y         = b2[e] + sum_kb sh[kb]*s2[e,n/128,kb] * (hq . w2[e,n])_kb
 *   out[t,:]    = bf16( sum_j w[t,j] * y[t,j,:] )    (slot order, no atomics)
 *
 * Padding rule (sizes that are not multiples of 128, e.g. 2880):
 *   Hp = ceil(H/128)*128, Ip = ceil(I/128)*128.  Logically w13 is
 *   [E, 2*Ip, Hp] e4m3 with gate rows at [0, I) and up rows at [Ip, Ip+I), and
 *   w2 is [E, Hp, Ip]; every padded row/column holds code 0; block scales
 *   cover the padded 128x128 blocks.  In memory the codes are BLOCKED: each
 *   128x128 block is 16 KB contiguous (row-major inside), blocks ordered
 *   [expert][row block][column block], i.e. w13 is [E, 2*Ip/128, Hp/128,
 *   128, 128] and w2 is [E, Hp/128, Ip/128, 128, 128], so a GEMM tile is one
 *   contiguous HBM read.  moe_pack_weights builds this layout.
 *
 * Ownership: the caller owns every buffer, including the workspace.  Calls
 * never allocate device memory, never synchronise the stream (except the two
 * status readers), keep no data between calls and are asynchronous on
 * `stream`.  Inputs are read-only; `out` is fully overwritten.  One exception:
 * moe_forward_static_scratch (below) uses a device array inside the library
 * instead of a workspace; that array lives until the process exits and keeps
 * the last call's contents.
 *
 * Errors: arguments are checked before any launch (MOE_ERR_INVALID_ARG,
 * MOE_ERR_UNSUPPORTED for pointers that are not 16-byte aligned or sizes
 * beyond the limits below, MOE_ERR_WORKSPACE for a short workspace); a failed
 * launch returns MOE_ERR_CUDA.  Every device-side wait is bounded (about 2 s);
 * a wait that runs out stops the kernel cleanly and sets an error word in
 * the workspace, which moe_read_device_status reports as
 * MOE_ERR_DEVICE_TIMEOUT.
 *
 * Limits: 1 <= top_k <= min(E, 8); 1 <= E <= 256; 1 <= T; T*top_k < 2^31;
 * 1 <= H, I <= 16384.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED = 2,
    MOE_ERR_WORKSPACE = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_DEVICE_TIMEOUT = 5
} moe_status;

/* Byte offsets of the intermediates inside the workspace (R = T*top_k).
 * After moe_forward completes they hold that call's values; tests read them. */
typedef struct {
    size_t total_bytes;
    size_t status;     /* uint32[64]: [0] device error word, [1] tile total GEMM1, [2] tile total GEMM2,
                          [3] rows per M tile */
    size_t hist;       /* int32 [ceil(T/256), E] tokens per (256-token chunk, expert), then 1 arrival counter */
    size_t count;      /* int32 [E]     rows per expert */
    size_t offset;     /* int32 [E+1]   first row of each expert (exclusive scan of count) */
    size_t chunk_base; /* int32 [ceil(T/256), E] first row of each (chunk, expert) */
    size_t tiles1;     /* int32 [E+1]   first gate/up GEMM tile of each expert */
    size_t tiles2;     /* int32 [E+1]   down GEMM tiles before each expert: its n-tiles per m-tile times
                          the m-tiles of the experts before it (a count prefix; at decode sizes the
                          kernel lists every m-tile's two-block tiles before the one-block ones) */
    size_t topk_idx;   /* int32 [T, top_k] selected experts, ascending */
    size_t topk_w;     /* float [T, top_k] softmax weights before bf16 rounding */
    size_t topk_wb;    /* bf16  [T, top_k] routing weights used by the layer */
    size_t perm;       /* int32 [R] row r -> t*top_k + j; rows sorted by (expert, token) */
    size_t inv;        /* int32 [R] t*top_k + j -> row */
    size_t xq;         /* e4m3  [R, Hp] quantised x, permuted rows */
    size_t sx;         /* float [Hp/128, R] group scales of xq, K-block-major */
    size_t hq;         /* e4m3  [R, Ip] requantised h */
    size_t sh;         /* float [Ip/128, R] group scales of hq, K-block-major */
    size_t part;       /* float [R, Hp] w[t,j]*y rows, indexed by t*top_k + j */
} moe_workspace_layout;

/* Bytes of workspace moe_forward needs for these sizes (0 if the sizes are invalid). */
size_t moe_workspace_size(int T, int H, int I, int E, int top_k);

/* Fills *layout for these sizes. */
moe_status moe_get_workspace_layout(int T, int H, int I, int E, int top_k, moe_workspace_layout* layout);

/*
 * The layer forward.
 *   x        bf16 [T, H] row-major          router_w bf16 [E, H]    router_b bf16 [E]
 *   w13      e4m3 blocked [E, 2*Ip/128, Hp/128, 128, 128]   s13 fp32 [E, 2*Ip/128, Hp/128]
 *   b13      bf16 [E, 2*I]  (gate [0,I), up [I,2I))
 *   w2       e4m3 blocked [E, Hp/128, Ip/128, 128, 128]     s2  fp32 [E, Hp/128, Ip/128]
 *   b2       bf16 [E, H]
 *   out      bf16 [T, H]
 *   workspace: device buffer of at least moe_workspace_size(...) bytes, 256-byte aligned.
 * All pointers are device pointers; x, router_w, w13, w2 and out must be 16-byte
 * aligned, the workspace 256-byte aligned (else MOE_ERR_UNSUPPORTED).
 * stream is a cudaStream_t (NULL = legacy default stream).
 */
moe_status moe_forward(const void* x, const void* router_w, const void* router_b, const uint8_t* w13, const float* s13,
                       const void* b13, const uint8_t* w2, const float* s2, const void* b2, int T, int H, int I, int E,
                       int top_k, void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_forward with timing marks: events[0..5] are cudaEvent_t handles the
 * caller created; events[i] is recorded on `stream` just before stage i
 * (0 router, 1 permutation + x quantisation, 2 gate/up GEMM, 3 down GEMM,
 * 4 combine) and events[5] after the last stage.  Same kernels, same results.
 */
moe_status moe_forward_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                const float* s13, const void* b13, const uint8_t* w2, const float* s2, const void* b2,
                                int T, int H, int I, int E, int top_k, void* out, void* workspace,
                                size_t workspace_bytes, void* stream, void* const* events);

/*
 * moe_forward for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that may not call cudaMalloc/cudaFree themselves -- for example plugins
 * whose device memory is owned by a host framework's caching allocator or a
 * serving engine's fixed pool, or code that must keep allocation and the
 * synchronisation cudaFree implies out of its latency path.  Same arguments
 * and results as moe_forward, without the workspace: the library uses a
 * file-scope device array of 32 MiB (MOE_STATIC_SCRATCH_BYTES) instead, which
 * every GPU that loads the library holds until the process exits.
 *   - Null pointers and invalid sizes return MOE_ERR_INVALID_ARG; sizes whose
 *     moe_workspace_size exceeds 32 MiB are rejected with MOE_ERR_WORKSPACE,
 *     both before anything is launched.
 *   - The first call in a CUDA context (per device, with that device current)
 *     looks up the array's device address (cudaGetSymbolAddress); make that
 *     first call before any stream capture.  A new context on the device (for
 *     example after cudaDeviceReset) is noticed and the address looked up
 *     again on the next call.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents (each call clears what must start at zero itself).
 *     Calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race on it; serialise them.
 *   - A device wait that ran out is reported by moe_read_static_scratch_status,
 *     not by the call's return value; the next call clears it.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
moe_status moe_forward_static_scratch(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                      const float* s13, const void* b13, const uint8_t* w2, const float* s2,
                                      const void* b2, int T, int H, int I, int E, int top_k, void* out, void* stream);

/* moe_read_device_status for the array of moe_forward_static_scratch on the
 * current device: synchronises `stream`, then reads and clears the error word
 * the last call left there (MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_CUDA). */
moe_status moe_read_static_scratch_status(void* stream);

/*
 * Routing steps alone, into caller buffers ("GPT-OSS on Day 0", MoE section:
 * the routing kernel -- top-k, then softmax over the selected experts -- kept
 * separate from the expert GEMMs, whose inputs it groups by expert):
 *   topk_idx int32 [T, top_k]  selected experts, ascending, ties -> lower index
 *   topk_w   fp32  [T, top_k]  softmax over the k logits before bf16 rounding
 *   offset   int32 [E+1]       first permuted row of each expert
 *   perm     int32 [R]         row r -> t*top_k + j, rows sorted by (expert, token)
 *   xq       e4m3  [R, Hp]     1x128 FP8 codes of x in permuted rows (pad codes 0)
 *   sx       fp32  [Hp/128, R] their group scales, K-block-major (sx[g*R + r])
 * The same kernels as moe_forward's first two stages.  x, router_w and xq must
 * be 16-byte aligned, the workspace (moe_route_workspace_size bytes) 256-byte
 * aligned; errors as moe_forward.  Asynchronous on `stream`.
 */
size_t moe_route_workspace_size(int T, int H, int E, int top_k);
moe_status moe_route_debug(const void* x, const void* router_w, const void* router_b, int T, int H, int E, int top_k,
                           int32_t* topk_idx, float* topk_w, int32_t* offset, int32_t* perm, uint8_t* xq, float* sx,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Row-major FP8 weight codes -> the blocked layout the forward reads.  The
 * layer's weights are e4m3 codes with 128x128 block scales ("GPT-OSS on Day
 * 0", infrastructure decisions); a caller that holds them row-major,
 *   w13_rm [E, 2*Ip, Hp] (gate rows [0, I), up rows [Ip, Ip+I), zero padding)
 *   w2_rm  [E, Hp, Ip]
 * gets w13 [E, 2*Ip/128, Hp/128, 128, 128] and w2 [E, Hp/128, Ip/128, 128,
 * 128] (each 128x128 block 16 KB contiguous).  The block scales s13 / s2 are
 * the same in both layouts and are not touched.  Also valid for MXFP8 codes
 * (same code layout).  All pointers 16-byte aligned device pointers; either
 * pair may be NULL to convert only the other.  Asynchronous on `stream`.
 */
moe_status moe_block_weights(const uint8_t* w13_rm, const uint8_t* w2_rm, int H, int I, int E, uint8_t* w13,
                             uint8_t* w2, void* stream);

/*
 * Weight packer (the offline converter from master weights to the layer's
 * FP8 layout; "GPT-OSS on Day 0": FP8 with 128x128 block scaling).
 *   w13_f32 fp32 [E, 2*I, H] (gate rows then up rows), w2_f32 fp32 [E, H, I]  (device)
 *   -> w13 e4m3 blocked [E, 2*Ip/128, Hp/128, 128, 128], s13 [E, 2*Ip/128, Hp/128],
 *      w2 e4m3 blocked [E, Hp/128, Ip/128, 128, 128], s2 [E, Hp/128, Ip/128]
 * Each 128x128 block: s = amax/448 (1 when the block is all zero), code =
 * e4m3_rne_satfinite(w/s) in IEEE fp32; padding gets code 0.
 * Either input may be NULL to pack only the other matrix.
 */
moe_status moe_pack_weights(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13, float* s13,
                            uint8_t* w2, float* s2, void* stream);

/*
 * The 1x128 group quantiser on its own (the step the gate/up GEMM epilogue
 * applies to h, and the one applied to x): in fp32 [rows, cols] with row
 * stride ld_in (elements) -> q e4m3 [rows, ceil(cols/128)*128],
 * s fp32 [rows, ceil(cols/128)].  It shares the per-value steps with the
 * fused epilogues -- the scale amax/448, its reciprocal, the corrected
 * quotient (IEEE division for groups with 0 < amax < 2^-64) and the e4m3
 * conversion -- but not the way they find a group's amax: the decode
 * epilogue takes a column maximum across a warp and switches the whole warp
 * to IEEE division when any of its tokens needs it, and the prefill epilogue
 * joins two warps' partial maxima through shared memory.
 */
moe_status moe_quantize_rows(const float* in, int rows, int cols, int ld_in, uint8_t* q, float* s, void* stream);

/*
 * MXFP8 variant.  "Hosting Qwen on Blackwell" (section "Quantization"): on
 * Blackwell, FP8 reaches full tensor-core throughput with microscaling, one
 * power-of-two scale per 32 consecutive values.  The layer above with every
 * 128x128 / 1x128 quantiser replaced by the OCP MX v1.0 (section 6.3) one:
 *   for a group of 32 values with absolute maximum amax
 *     X    = floor(log2(amax)) - 8, clamped to [-127, 127]; scale byte X + 127 (UE8M0)
 *     code = e4m3_rne_satfinite(v * 2^-X)    (an all-zero group: byte 0, +0 codes)
 *   x and h in groups of 32 along the row (H, I), weights along K per output row;
 *   acc = bias + sum_g 2^(sa_g - 127) * 2^(sw_g - 127) * (xq . w)_g, fp32 accumulation.
 * Same padding (Hp, Ip) and the same blocked code layout as the 128x128
 * variant.  Scales are bytes in 512-byte ATOMS: one atom per 128x128 code
 * block, holding that block's 128 rows x 4 groups, byte (r % 32) * 16 +
 * (r / 32) * 4 + g for row r and group g (the layout the tensor core reads
 * after tcgen05.cp 32x128b.warpx4):
 *   s13 uint8 [E, 2*Ip/128, Hp/128, 512]     s2 uint8 [E, Hp/128, Ip/128, 512]
 * Padding rows and columns get byte 0 and code 0.
 */

/* Workspace of moe_forward_mx (the same fields as moe_workspace_layout, except
 * that sx and sh hold scale atoms: [m-tiles, Hp/128, 512] and [m-tiles,
 * Ip/128, 512], where the rows of expert e form m-tiles of bm rows from
 * offset[e] -- bm = 32 when T*top_k <= 64*E, else 128 -- and expert e's
 * m-tiles are numbered from tiles1[e] / (Ip/128)). */
size_t moe_workspace_size_mx(int T, int H, int I, int E, int top_k);
moe_status moe_get_workspace_layout_mx(int T, int H, int I, int E, int top_k, moe_workspace_layout* layout);

/*
 * The MXFP8 layer forward.  Arguments as moe_forward, except s13 and s2: the
 * scale atoms above (device, 16-byte aligned).  The workspace is sized by
 * moe_workspace_size_mx.
 */
moe_status moe_forward_mx(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                          const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2, const void* b2,
                          int T, int H, int I, int E, int top_k, void* out, void* workspace, size_t workspace_bytes,
                          void* stream);

/* moe_forward_mx with the timing marks of moe_forward_profiled. */
moe_status moe_forward_mx_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                   const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2,
                                   const void* b2, int T, int H, int I, int E, int top_k, void* out, void* workspace,
                                   size_t workspace_bytes, void* stream, void* const* events);

/*
 * MXFP8 weight packer: fp32 masters (as moe_pack_weights) -> blocked e4m3
 * codes and scale atoms.  Every output row is quantised along K in groups of
 * 32.  All output pointers 16-byte aligned; either input may be NULL.
 */
moe_status moe_pack_weights_mx(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13,
                               uint8_t* s13, uint8_t* w2, uint8_t* s2, void* stream);

/*
 * The 1x32 MX quantiser on its own: in fp32 [rows, cols], row stride ld_in
 * -> q e4m3 [rows, cp], s uint8 [rows, cp/32] row-major, cp = cols padded to
 * a multiple of 128 (padding groups: byte 0, codes 0).  Same device
 * arithmetic as the MX kernels' quantisers.
 */
moe_status moe_quantize_rows_mx(const float* in, int rows, int cols, int ld_in, uint8_t* q, uint8_t* s,
                                void* stream);

/* ---------------------------------------------------------------------------
 * MXFP4 weights.  "GPT-OSS on Day 0" (opening section): the open-weight
 * models ship with MXFP4 weights, which Blackwell's FP4 tensor cores run
 * natively; "Hosting Qwen on Blackwell" (section "Quantization") names the
 * microscaled formats as the fast path there.  Weights are OCP MX v1.0 FP4
 * E2M1 codes (section 5.3.3: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, sign in
 * bit 3) with one UE8M0 scale per 32 values along K, shared exponent
 * floor(log2(amax)) - 2 (section 6.3); x and h stay MXFP8 exactly as in
 * moe_forward_mx.  The codes are packed two per byte, value 2j in the low
 * nibble of byte j, each 128 x 128 block contiguous (64-byte rows):
 *   w13 uint8 [E, 2*Ip/128, Hp/128, 128, 64]   w2 uint8 [E, Hp/128, Ip/128, 128, 64]
 * the scale atoms are those of the MXFP8 layout.  Half the weight bytes of
 * the e4m3 formats.
 * ------------------------------------------------------------------------- */

/*
 * The layer with MXFP4 weights.  Arguments as moe_forward_mx, with w13 and w2
 * in the packed layout above (device, 32-byte aligned, else
 * MOE_ERR_UNSUPPORTED).  The workspace is sized by moe_workspace_size_mx.
 */
moe_status moe_forward_mxfp4(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                             const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2, const void* b2,
                             int T, int H, int I, int E, int top_k, void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* moe_forward_mxfp4 with the timing marks of moe_forward_profiled. */
moe_status moe_forward_mxfp4_profiled(const void* x, const void* router_w, const void* router_b, const uint8_t* w13,
                                      const uint8_t* s13, const void* b13, const uint8_t* w2, const uint8_t* s2,
                                      const void* b2, int T, int H, int I, int E, int top_k, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream, void* const* events);

/*
 * MXFP4 weight packer: fp32 masters (as moe_pack_weights) -> packed E2M1
 * codes (nearest, ties to the even code, magnitudes above 6 * 2^X saturate)
 * and scale atoms.  An all-zero group gets byte 0 and +0 codes; padding rows
 * and columns are zero.  Output pointers 16-byte aligned (32 for use by
 * moe_forward_mxfp4); either input may be NULL.
 */
moe_status moe_pack_weights_mxfp4(const float* w13_f32, const float* w2_f32, int H, int I, int E, uint8_t* w13,
                                  uint8_t* s13, uint8_t* w2, uint8_t* s2, void* stream);

/* Synchronises `stream`, then reads and clears the device error word of
 * `workspace`: MOE_OK, MOE_ERR_DEVICE_TIMEOUT (a bounded wait ran out), or
 * MOE_ERR_CUDA. */
moe_status moe_read_device_status(void* workspace, void* stream);

/*
 * Check of the bounded-wait machinery: one thread waits on a barrier that
 * receives `arrivals` arrivals out of the 1 it needs (0 = never completes),
 * for at most timeout_ns.  Writes 1 (completed) or 2 (timed out) to
 * *result_dev (device uint32).  No fault, trap or hang is possible.
 */
moe_status moe_test_bounded_wait(uint64_t timeout_ns, int arrivals, uint32_t* result_dev, void* stream);

const char* moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
