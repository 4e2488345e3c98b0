// internal.h -- host-side declarations shared by the libmbw translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "mbw.h"

namespace mbw {

enum Fmt : int { FMT_BF16 = 0, FMT_G64 = 1, FMT_AWQ = 2, FMT_I8 = 3 };

// Arguments of one weight-streaming GEMV launch. A "chunk" is 16 bytes of one
// weight row: 8 bf16 weights, 32 INT4 codes or 16 INT8 codes.
struct GemvArgs {
    const uint8_t* W;        // weight rows, `chunks` 16-byte chunks each
    const uint16_t* scales;  // fp16 group scales [N][groups] (INT4 only)
    const uint8_t* zeros;    // packed uint4 zero points [N][zstride] (AWQ only)
    const uint16_t* x;       // bf16 activations [M][K]
    void* y;                 // bf16 or fp32 outputs [M][N]
    int N, K, M;
    int chunks;        // 16-byte chunks per weight row
    int split_chunks;  // chunks handled by one CTA of a split-K cluster
    int groups;        // scale groups per row
    int zstride;       // zero-point bytes per row
    int out_f32;       // 1: write fp32 y
    const float* rscale;  // fp32 scale per weight row [N] (INT8 only)
    // Fusions (NULL / 0 = none). RMSNorm prologue: x <- bf16(x * norm_w / sqrt(mean(x^2) + eps)).
    const uint16_t* norm_w;  // bf16 [K]
    float norm_eps;
    // Residual epilogue: y <- y + residual (bf16 [M][N]; may be y itself).
    const uint16_t* residual;
    // Gated epilogue: W2 (+ scales2 / rscale2) is the "up" matrix of the same shape and format;
    // y <- silu(W.x) * (W2.x). Its tiles interleave with W's: logical tile 2p is W's tile p, 2p+1 is W2's.
    int glu;
    const uint8_t* W2;
    const uint16_t* scales2;
    const float* rscale2;
    const uint8_t* zeros2;  // the up matrix's zero points (AWQ)
    // INT4 codes in the load-time repacked layout (mbw_repack_int4): the
    // unpack then yields the k pairs in natural order, and x is staged as is
    // instead of with the pair permutation.
    int x_natural;
};

// Logical 16-row tiles of a launch (twice the output tiles under the gated epilogue).
inline int64_t gemv_tiles(int64_t N, int glu) { return (N + 15) / 16 * (glu ? 2 : 1); }
// 1 if the launch uses a fusion (it then runs the kernels' FZ = 1 instantiations).
inline int gemv_fused_args(const GemvArgs& a) { return (a.glu || a.norm_w || a.residual) ? 1 : 0; }

// One instantiation of the CUDA-core streaming kernel.
struct SimtConfig {
    int warps;  // warps per CTA, each owning its own rows
    int r;      // rows per warp, streamed together
    int u;      // chunks per lane per row in flight
    int mb;     // activation rows (batch) per launch
    int cb;     // bytes per lane per load: 16, or 32 (BF16 batch 1: a warp reads 1 KB of a row per load)
    int persist = 0;  // 32-byte BF16 only: occ CTAs per SM loop over the row groups (no split)
};

// One instantiation of the tensor-core (mma.sync) streaming kernel.
struct MmaConfig {
    int warps;  // warps per CTA; each owns one k-slice of every tile of the CTA
    int u;      // row blocks per lane in flight (ring depth)
    int async;  // 1: the ring lives in shared memory, filled with cp.async
};

// One instantiation of the latency-oriented kernel (whole share in registers
// before the wait).
struct LatConfig {
    int warps;   // warps per CTA
    int wt;      // warps along the CTA's row tiles (the other warps / wt split K)
    int ni;      // most items (16 rows x one 128-byte super-block) a warp may own
    int npre;    // items unpacked to MMA fragments before the wait (INT4)
    int staged;  // 1: items past npre wait in a shared-memory ring (cp.async), not registers
    int lean;    // 1: unpack and MMA one 32-bit word at a time from the ring (few registers)
};

// One instantiation of the bulk-copy-fed tensor-core streaming kernel.
struct TmaConfig {
    int warps;  // consumer warps per CTA (plus one producer warp)
    int depth;  // shared-memory ring stages
};

// One instantiation of the BF16 row-stream kernel (gemv_tma.cu): per-warp
// bulk-copy rings over the CTA's contiguous rows.
struct RowsConfig {
    int warps;  // warps per CTA, each with its own ring and copy-issuing lane
    int depth;  // ring slots per warp
    int seg;    // bytes per stage (one bulk copy)
};

// One instantiation of the bulk-fed INT4 kernel (gemv_tma.cu): a producer
// lane fills a CTA ring of 16-row stages for W consumer warps.
struct QbulkConfig {
    int warps;  // consumer warps (plus one producer warp)
    int depth;  // ring stages
    int bsc;    // super-blocks per consumer warp per stage
};

// One instantiation of the batched AWQ mma.sync kernel (gemv_awq_batch.cu).
struct AwqbConfig {
    int nb;    // n-blocks of 8 batch rows (the launch covers up to 8 * nb rows)
    int wt;    // warps along the CTA's tiles (warp (wt, wk) owns tiles wt, wt + WT, ...)
    int wk;    // warps along the CTA's k-range (each an even share of its super-blocks)
    int u;     // super-blocks (256 k) per lane in flight (register ring depth)
    int minb;  // CTAs per SM its register budget allows (at most this many per SM)
    int early; // 1: a ring slot is refilled before its super-block is computed
    int async; // 1: the ring is in shared memory (cp.async), scales and zero points in per-CTA tables
    int fmt;   // FMT_AWQ, or FMT_I8 (symmetric INT8 with a per-row scale, batches above 8)
};

// Execution plan of one call shape.
struct Plan {
    int kind;   // PLAN_SIMT or PLAN_MMA
    int cfg;    // index into the kernel table of `kind`
    int split;  // CTAs per cluster along K (1 = no split)
    int occ;    // MMA kernels: CTAs per SM in the persistent grid (1 for SIMT)
};
enum PlanKind : int {
    PLAN_NONE = -1,  // no kernel fits the shape (the call returns MBW_ERR_UNSUPPORTED)
    PLAN_SIMT = 0,
    PLAN_MMA = 1,
    PLAN_TMA = 2,
    PLAN_MMA2 = 3,
    PLAN_TC = 4,
    PLAN_LAT = 5,
    PLAN_AWQB = 6,
    PLAN_ROWS = 7,
    PLAN_QBULK = 8,
};

// Kernel tables (gemv_simt.cu).
int simt_num_configs(int fmt);
SimtConfig simt_config(int fmt, int idx);
cudaError_t launch_gemv_simt(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);
size_t simt_smem_bytes(int fmt, const SimtConfig& c, const GemvArgs& a, int split);

// Tensor-core kernel tables (gemv_mma.cu).
int mma_num_configs(int fmt);
MmaConfig mma_config(int fmt, int idx);
int mma_max_batch(int fmt);
size_t mma_smem_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ);
int mma_row_groups(int64_t N, int split, int occ);
cudaError_t launch_gemv_mma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);

// Shared memory a GEMV launch may ask for (the planner's limit).
constexpr size_t kSmemFit = 200 * 1024;

// CTA row-groups of a launch whose shared memory holds the partial sums of
// every 16-row tile a CTA owns: the one-wave count of mma_row_groups when that
// layout fits `limit` bytes, else the fewest groups whose layout does (a very
// tall matrix then runs in several waves; its CTAs depend on no CTA outside
// their own cluster). bytes(G), the layout's size for G groups, never grows
// with G; when not even one tile per CTA fits, the one-wave count is returned
// and the caller's size check refuses the plan.
template <class F>
int fitted_row_groups(int64_t N, int split, int occ, size_t limit, F bytes) {
    const int64_t G = mma_row_groups(N, split, occ);
    const int64_t T = (N + 15) / 16;
    if (G >= T || bytes((int)G) <= limit || bytes((int)T) > limit) return (int)G;
    int64_t lo = G + 1, hi = T;  // bytes(hi) fits
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (bytes((int)mid) <= limit)
            hi = mid;
        else
            lo = mid + 1;
    }
    return (int)lo;
}

// 32-bytes-per-lane tensor-core kernel tables (gemv_mma.cu).
int mma2_num_configs(int fmt);
MmaConfig mma2_config(int fmt, int idx);
int mma2_max_batch(int fmt);
int mma2_block_k(int fmt);
size_t mma2_smem_bytes(int fmt, const MmaConfig& c, int64_t N, int64_t K, int M, int split, int occ, int glu = 0);
cudaError_t launch_gemv_mma2(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);

// Latency-oriented kernel tables (gemv_lat.cu).
int lat_num_configs(int fmt);
LatConfig lat_config(int fmt, int idx);
int lat_max_batch(int fmt);
int lat_block_k(int fmt);
int lat_items_per_warp(int fmt, const LatConfig& c, int64_t N, int64_t K, int split, int occ, int glu = 0);
size_t lat_smem_bytes(int fmt, const LatConfig& c, int64_t N, int64_t K, int M, int split, int occ, int glu = 0,
                      int fz = 0);
cudaError_t launch_gemv_lat(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);

// Batched AWQ mma.sync kernel tables (gemv_awq_batch.cu): batches of 5 .. 64
// rows per launch, K % 256 == 0.
int awqb_num_configs();
AwqbConfig awqb_config(int idx);
int awqb_row_groups(const AwqbConfig& c, int64_t N, int64_t K, int split, int occ);
size_t awqb_smem_bytes(const AwqbConfig& c, int64_t N, int64_t K, int split, int occ);
cudaError_t launch_gemv_awq_batch(const Plan& p, const GemvArgs& a, cudaStream_t s);

// tcgen05 skinny GEMM (gemm_tc.cu): Y = X . W^T for the whole batch M.
// cfg bit 0: ring (0 deep, 1 co-resident); bit 1: two 64-k boxes per stage
cudaError_t launch_gemm_tc(const uint16_t* X, const uint16_t* W, void* Y, int64_t M, int64_t N, int64_t K, int split,
                           int cfg, int out_f32, cudaStream_t s);
int tc_batch_tile(int64_t M);
// tcgen05 AWQ-style INT4 batched GEMM (gemm_tc.cu): whole batch M, slices of 64.
// x_natural: the codes are in the repacked layout (no X permutation).
cudaError_t launch_gemm_tc_awq(const uint8_t* Q, const uint16_t* scales, const uint8_t* zeros, const uint16_t* X,
                               void* Y, int64_t M, int64_t N, int64_t K, int split, int out_f32, int x_natural,
                               cudaStream_t s);
int tc_awq_batch_tile(int64_t M);
bool tc_awq_fits(int64_t M, int64_t K, int split);  // the split leaves room for the scale/zero tables
int tc_take_fault();
cudaError_t launch_tc_wait_expiry(long long tries, cudaStream_t s);  // a bounded wait that expires

// Bulk-copy-fed kernel tables (gemv_tma.cu).
int tma_num_configs(int fmt);
TmaConfig tma_config(int fmt, int idx);
size_t tma_smem_bytes(int fmt, const TmaConfig& c, int64_t N, int64_t K, int M, int split, int occ);
cudaError_t launch_gemv_tma(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);
int rows_num_configs();
RowsConfig rows_config(int idx);
int rows_ctas(int64_t N, int occ);
size_t rows_smem_bytes(const RowsConfig& c, int64_t N, int64_t K, int occ);
cudaError_t launch_gemv_rows(const Plan& p, const GemvArgs& a, cudaStream_t s);
int qbulk_num_configs(int fmt);
QbulkConfig qbulk_config(int fmt, int idx);
size_t qbulk_smem_bytes(int fmt, const QbulkConfig& c, int64_t N, int64_t K, int M, int split, int occ);
cudaError_t launch_gemv_qbulk(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);
int tma_take_fault();  // 1 if a bounded device wait expired since the last call (and clear it)
cudaError_t launch_tma_wait_expiry(long long tries, cudaStream_t s);  // a bounded wait that expires

cudaError_t launch_dequant(int fmt, const uint8_t* Wq, const uint16_t* scales, const uint8_t* zeros,
                           float* out, int64_t N, int64_t K, cudaStream_t s);
// INT8 load-time quantizer (quantize.cu).
cudaError_t launch_quantize_int8_pc(const uint16_t* W, int8_t* Wq, float* scales, int64_t N, int64_t K,
                                    cudaStream_t s);
// Load-time INT4 repack (quantize.cu): N x K/8 words, in place allowed.
cudaError_t launch_repack_int4(const uint8_t* Wq, uint8_t* Wr, int64_t N, int64_t K, cudaStream_t s);

// Plan cache (plan.cu).
Plan plan_lookup(int op, int64_t M, int64_t N, int64_t K, cudaStream_t s);
Plan plan_default(int op, int64_t M, int64_t N, int64_t K);
std::string plan_to_string(int op, const Plan& p);
int plan_batch_width(int fmt, const Plan& p);  // activation rows per launch
cudaError_t launch_plan(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s);

// Error reporting (abi.cu).
void set_last_error(const std::string& msg);
void count_launch();
int device_sm_count();

}  // namespace mbw
