// Host-side launch wrappers and parameter blocks shared by the library's
// translation units (not part of the public C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

struct RouteParams {
    const uint16_t* x;   // bf16 [T, H]
    const uint16_t* rw;  // bf16 [E, H]
    const uint16_t* rb;  // bf16 [E]
    int T, H, E, k;
    int nchunks;  // ceil(T / kChunkTokens)
    int nt1, nt2; // n-tiles per M tile: gate/up GEMM (Ip/128), down GEMM (Hp/128)
    int bm;       // rows per M tile: 128 (prefill kernels) or 32 (decode kernels)
    int32_t* topk_idx;
    float* topk_w;
    uint16_t* topk_wb;
    int32_t* hist;    // [nchunks, E], zeroed before the launch
    int32_t* done;    // arrival counter of finished router CTAs, zeroed before the launch: the last
                      // one scans the histogram into count, offset, chunk_base and the tile lists,
                      // which are final when the router grid completes (the GEMMs read them before
                      // they wait for the permutation kernel)
    int32_t* count;
    int32_t* offset;
    int32_t* chunk_base;
    int32_t* tiles1;
    int32_t* tiles2;
    uint32_t* status;
};

struct PermuteParams {
    const uint16_t* x;
    int T, H, Hp, E, k;
    int tokens_per_cta;
    int early_dependents;  // set at launch: 1 when the grid is one wave (the next kernel may start early)
    const int32_t* topk_idx;
    const int32_t* chunk_base;
    int bm, nt1;
    const int32_t* offset;  // MXFP8: first row and first m-tile of each expert (scale atom positions)
    const int32_t* tiles1;
    int32_t* perm;
    int32_t* inv;
    int R;        // T * k
    uint8_t* xq;  // [R, Hp]
    float* sx;    // [Hp/128, R] (K-block-major)
    // MXFP8 variant: 1x32 UE8M0 scales into scale atoms [m-tiles, Hp/128, 512]
    // (m-tile of row r of expert e: tiles1[e]/nt1 + (r - offset[e])/bm)
    int mx;
    uint8_t* sxa;
};

constexpr int kDecXBoxRows = 8;  // activation rows per TMA box of the decode GEMMs
#ifndef MOE_DEC_STAGES_GATEUP
#define MOE_DEC_STAGES_GATEUP 5
#endif
#ifndef MOE_DEC_STAGES_DOWN
#define MOE_DEC_STAGES_DOWN 9
#endif
// K blocks per ring stage of the MX decode GEMMs: the down GEMM (one weight
// block per K block) runs faster with two per stage (oss120b_decode: MXFP8
// 209 -> 186 us, MXFP4 210 -> 182 us), the gate/up GEMM slower (326 -> 344,
// 274 -> 285 us)
#ifndef MOE_MX_DEC_KPS_GATEUP
#define MOE_MX_DEC_KPS_GATEUP 1
#endif
#ifndef MOE_MX_DEC_KPS_DOWN
#define MOE_MX_DEC_KPS_DOWN 2
#endif
// K blocks per ring stage of the 128x128 decode GEMMs (two were slower for both)
#ifndef MOE_DEC_KPS_GATEUP
#define MOE_DEC_KPS_GATEUP 1
#endif
#ifndef MOE_DEC_KPS_DOWN
#define MOE_DEC_KPS_DOWN 1
#endif
constexpr int kDecStagesGateUp = MOE_DEC_STAGES_GATEUP;  // stage ring depth of the decode GEMMs (upper bound)
constexpr int kDecStagesDown = MOE_DEC_STAGES_DOWN;

struct GemmParams {
    int E, R, KB;          // K / 128
    int N_real;            // gate/up GEMM: I; down GEMM: H
    int rows_B;            // rows of one expert's weight matrix: 2*Ip or Hp
    int up_rows;           // rows from a tile's first weight row block to its second: gate/up GEMM Ip
                           // (the up half); paired decode down GEMM ceil(Hp/256)*128; else 0
    int sw_rowblocks;      // rows_B / 128
    const int32_t* count;
    const int32_t* offset;
    const int32_t* tiles;  // [E+1] first tile of each expert
    const float* sa;       // activation scales [KB, R] (K-block-major)
    const float* sw;       // weight scales [E, rows_B/128, KB]
    const uint16_t* bias;  // gate/up: b13 [E, 2I]; down: b2 [E, H]
    uint8_t* hq;           // gate/up output codes [R, ldq]
    float* sh;             // gate/up output scales [ldq/128, R] (K-block-major)
    int ldq;
    const int32_t* perm;      // down: row -> t*k + j
    const uint16_t* topk_wb;  // down: routing weights bf16 [T*k]
    float* part;              // down: [T*k, ldp]
    int ldp;
    uint32_t* status;
};

// The MXFP8 GEMMs: scales are UE8M0 bytes in 512-byte atoms (one per 128
// rows x one 128-wide K block, mx_atom_byte layout); the tile list is the same
// as the 128x128 variant's.
struct MxGemmParams {
    int E, R, KB;          // K / 128
    int N_real;            // gate/up GEMM: I; down GEMM: H
    int sw_rowblocks;      // rows of one expert's weight matrix / 128
    int up_rows;           // rows from a tile's first weight row block to its second: gate/up GEMM Ip
                           // (the up half); paired decode down GEMM ceil(Hp/256)*128; else 0
    int nt;                // n-tiles per m-tile (tiles[e] = nt * m-tiles of the experts before e)
    const int32_t* count;
    const int32_t* offset;
    const int32_t* tiles;  // [E+1] first tile of each expert
    const uint8_t* sa;     // activation scale atoms [m-tiles, KB, 512]
    const uint8_t* sw;     // weight scale atoms [E, sw_rowblocks, KB, 512]
    const uint16_t* bias;  // gate/up: b13 [E, 2I]; down: b2 [E, H]
    uint8_t* hq;           // gate/up output codes [R, ldq]
    uint8_t* sh;           // gate/up output scale atoms [m-tiles, ldq/128, 512]
    int ldq;
    const int32_t* perm;      // down: row -> t*k + j
    const uint16_t* topk_wb;  // down: routing weights bf16 [T*k]
    float* part;              // down: [T*k, ldp]
    int ldp;
    uint32_t* status;
};

// Launch with programmatic stream serialisation allowed (the kernel calls
// griddepcontrol.wait before reading what earlier kernels wrote).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_router(const RouteParams& p, cudaStream_t st);
// Tensor-core router: the padded expert count NP it would use (32, 64, 128 or
// 256), or 0 when the layer takes the cluster kernel above (fewer than 2048
// tokens, rows not 16-byte aligned, more than 256 experts).  tmX / tmW are
// bf16 tensor maps of x [T, H] and the router weights [E, H] with 64 x 128 and
// 64 x NP boxes (128-byte swizzle).
int router_tc_experts(int T, int H, int E);
cudaError_t launch_router_tc(const RouteParams& p, const CUtensorMap& tmX, const CUtensorMap& tmW, cudaStream_t st);
cudaError_t launch_permute_quant(const PermuteParams& p, cudaStream_t st);
cudaError_t launch_combine(const float* part, int T, int H, int ldp, int k, uint16_t* out, int num_sms,
                           cudaStream_t st);
cudaError_t launch_pack_blocks(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p, int gated_I,
                               uint8_t* q, float* s, cudaStream_t st);
cudaError_t launch_quantize_rows(const float* in, int rows, int cols, int ld_in, uint8_t* q, float* s,
                                 cudaStream_t st);
cudaError_t launch_pack_blocks_mx(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p, int gated_I,
                                  uint8_t* q, uint8_t* s, cudaStream_t st);
cudaError_t launch_pack_blocks_mx4(const float* src, int E, int rows_src, int cols, int rows_p, int cols_p,
                                   int gated_I, uint8_t* q, uint8_t* s, cudaStream_t st);
cudaError_t launch_quantize_rows_mx(const float* in, int rows, int cols, int ld_in, uint8_t* q, uint8_t* s,
                                    cudaStream_t st);
// Row-major codes [E, rows, cols] (rows, cols multiples of 128) -> blocked
// [E, rows/128, cols/128, 128, 128]; 16-byte aligned pointers.
cudaError_t launch_block_codes(const uint8_t* src, int E, int rows, int cols, uint8_t* dst, cudaStream_t st);
cudaError_t launch_bounded_wait_test(uint64_t timeout_ns, int arrivals, uint32_t* result, cudaStream_t st);
cudaError_t launch_gemm_gateup(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                               cudaStream_t st);
cudaError_t launch_gemm_down(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                             cudaStream_t st);
cudaError_t launch_gemm_gateup_decode(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p, int grid,
                                      cudaStream_t st);
cudaError_t launch_gemm_down_decode(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmParams& p, int grid,
                                    cudaStream_t st);

// tmX: activation rows (prefill: 128-row boxes, decode: kDecXBoxRows-row boxes); tmW: blocked weights
// fp4w: the weight codes are E2M1 (MXFP4), loaded through a 16U4_ALIGN16B tensor map.
cudaError_t launch_gemm_mx(bool gated, bool decode, bool fp4w, const CUtensorMap& tmX, const CUtensorMap& tmW,
                           const MxGemmParams& p, int grid, cudaStream_t st);

}  // namespace moe
