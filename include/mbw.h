/*
 * mbw.h -- C ABI of libmbw.so: the decode-step weight-streaming matrix-vector
 * product on GB300 (sm_103a).
 *
 * The operation (the one all the pages turn on):
 *   y = W . x, W stored (N, K) row-major, x of length K, y of length N: one
 *   output per weight row, "W (d,n) @ x (n,) -> xout (d,)" (yalm, "Fast LLM
 *   inference from scratch", sec. 2 CPU matmul and sec. 3.1 GPU matmul). In
 *   batch-1 decode every weight is read once per token and used for one
 *   multiply-add, so the call is bound by memory bandwidth (llm-rs vs vLLM,
 *   sec. 2 "Decode with one request is a memory problem"; tinyinfer, "How I
 *   Built an LLM Inference Engine From Scratch in CUDA", TL;DR).
 *   Batched: Y = X . W^T, X (M, K), Y (M, N): the same weights read once for M
 *   activation rows (llm-rs vs vLLM, sec. 3 "Batching moves decode from memory
 *   toward math").
 *
 * Conventions shared by every call below:
 *   - Pointers are device pointers on the current CUDA device, row-major and
 *     contiguous, 16-byte aligned (MBW_ERR_MISALIGNED otherwise); the weight
 *     (code) pointer W / Wq must be 32-byte aligned, because the kernels read
 *     weights with 256-bit loads. The caller owns every buffer; the library
 *     never allocates on a call path.
 *   - bf16 = IEEE bfloat16, fp16 = IEEE binary16, passed as raw bits.
 *   - Accumulation is fp32; the output is rounded to bf16 (round to nearest
 *     even) unless mbw_set_output_fp32(1) is in effect on the calling thread.
 *   - N == 0 or M == 0: nothing is launched, MBW_OK. K == 0: y is set to zero.
 *   - Calls are asynchronous on `stream`; arguments are checked on the host
 *     before any CUDA call and reported as a status, never thrown. Launch
 *     errors are returned as MBW_ERR_CUDA (detail in mbw_last_error()).
 *   - Shapes no kernel fits return MBW_ERR_UNSUPPORTED before any launch:
 *     the GEMV kernels stage the x of one CTA's k-range (split over at most
 *     8 CTAs of a cluster) in shared memory, so very long rows have no plan
 *     (batch 1: K above about 650,000 for INT8 and 800,000 for BF16 and INT4;
 *     wider batches proportionally less). gemm_skinny_bf16 from M = 5 on
 *     streams X through its tensor-core ring and takes any K.
 *     mbw_plan_candidates() == 0 tells in advance. Tall matrices have no such
 *     limit: a launch whose per-tile partial sums do not fit one wave of CTAs
 *     runs in several.
 *   - y must not alias an input. Results are deterministic: the same inputs
 *     give bitwise the same outputs, run after run.
 *   - Kernels use programmatic dependent launch: each GEMV/GEMM starts
 *     streaming W (and scales, zero points) before it waits for the previous
 *     kernel in the stream, and reads x only after that wait. So x may be
 *     produced by the preceding kernel, but the weights must not be: a kernel
 *     that writes weights must have completed before the GEMV is launched
 *     behind it. The library's own weight writers (mbw_quantize_int8_pc,
 *     mbw_repack_int4) see to this themselves: each ends with an empty kernel
 *     launched with plain stream ordering, which starts only after the writer
 *     has completed, so a GEMV queued next on the same stream reads the
 *     finished weights without a host synchronization.
 *   - `workspace` / `ws_bytes` are accepted for split-K plans that need global
 *     scratch; a NULL or short workspace never fails a call (the plan falls
 *     back to a variant that needs none). mbw_workspace_bytes() gives the size.
 *   - Threads: calls are thread-safe. The plan cache is shared and guarded.
 *     Calls can be captured into a CUDA graph once their shape is planned
 *     (mbw_autotune, or one earlier call); a shape first seen during capture
 *     uses the built-in default plan and is never autotuned there.
 */
#ifndef MBW_H
#define MBW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (a pointer to the driver's stream object).
 * NULL selects the legacy default stream. */
typedef struct CUstream_st *mbw_stream_t;

typedef int mbw_status;
#define MBW_OK 0
#define MBW_ERR_INVALID_ARG 1         /* NULL pointer, negative size, bad flag */
#define MBW_ERR_MISALIGNED 2          /* a pointer is not 16-byte aligned */
#define MBW_ERR_BAD_SHAPE 3           /* K not a multiple of the format's unit, sizes too large */
#define MBW_ERR_WORKSPACE_TOO_SMALL 4 /* only from calls that require scratch */
#define MBW_ERR_UNSUPPORTED 5         /* no kernel for this device or request */
#define MBW_ERR_CUDA 6                /* a CUDA runtime call failed */
#define MBW_ERR_DEVICE_TIMEOUT 7      /* a device-side bounded wait gave up */

/* Largest N, K or M a call accepts (MBW_ERR_BAD_SHAPE above it). The kernels
 * index rows and columns in 32-bit integers, and a tile may run up to 256 rows
 * past N before its clamp; the 2^16 of headroom keeps every such index
 * positive. */
#define MBW_MAX_DIM ((1LL << 31) - (1LL << 16))

/* Rounds of mbarrier.try_wait a kernel's wait makes before it gives up, sets
 * the device fault flag and leaves its loop (the waits of the bulk-copy and
 * tcgen05 kernels). A round that does not complete suspends for ~3.8 us on a
 * GB300, so a stalled wait gives up after about 1 s of running time; a wait
 * the pipeline satisfies lasts microseconds. */
#define MBW_WAIT_LIMIT (1LL << 18)

/* Operation ids for the plan / workspace queries. */
#define MBW_OP_GEMV_BF16 1
#define MBW_OP_GEMV_INT4_G64 2
#define MBW_OP_GEMV_INT4_AWQ_G128 3
#define MBW_OP_GEMM_SKINNY_BF16 4
#define MBW_OP_GEMV_INT8_PC 5
/* Fusion bits, or-ed into an op id for the plan queries of gemv_fused calls
 * (the bits follow the mbw_fusion fields that are set). */
#define MBW_OP_BASE_MASK 0xFF
#define MBW_FUSE_NORM 0x100     /* RMSNorm prologue */
#define MBW_FUSE_GLU 0x200      /* gated SiLU epilogue */
#define MBW_FUSE_RESIDUAL 0x400 /* residual-add epilogue */
#define MBW_FUSE_MASK 0x700
/* Plan-key flag of gemv_int4_awq_g128_repacked: codes in the repacked layout. */
#define MBW_REPACKED 0x800

/*
 * gemv_bf16 -- y = W . x with BF16 weights (16 bits per weight; llm-rs vs
 * vLLM, sec. 6 format table, "BF16 16").
 *   W : bf16 [N][K]      x : bf16 [K]      y : bf16 [N] (fp32 [N] under the fp32 hook)
 *   Requires K % 8 == 0 (16-byte rows). N, K <= MBW_MAX_DIM.
 */
mbw_status gemv_bf16(const void *W, const void *x, void *y, int64_t N, int64_t K,
                     void *workspace, size_t ws_bytes, mbw_stream_t stream);

/*
 * gemv_int4_g64 -- y = W . x with INT4 group-64 weights: 4-bit codes plus one
 * fp16 scale per 64 consecutive weights of a row (tinyinfer, TL;DR: "4 bits
 * plus one fp16 scale per 64 weights"), dequantized as w = (q - 8) * s.
 *   Wq     : uint8 [N][K/2], two codes per byte, low nibble = even k
 *   scales : fp16  [N][K/64]
 *   x      : bf16  [K]       y : bf16 [N] (fp32 under the fp32 hook)
 *   Requires K % 64 == 0. `scales` needs only 2-byte alignment.
 */
mbw_status gemv_int4_g64(const uint8_t *Wq, const void *scales, const void *x, void *y,
                         int64_t N, int64_t K, void *workspace, size_t ws_bytes,
                         mbw_stream_t stream);

/*
 * gemv_int4_awq_g128 -- Y = X . W^T with AWQ-style INT4 weights: 4-bit codes
 * with an fp16 scale and a 4-bit zero point per 128 consecutive weights of a
 * row (llm-rs vs vLLM, sec. 6 format table, "AWQ: 4-bit, FP16 scale + zero per
 * 128"), dequantized as w = (q - z) * s. M = 1 is the decode GEMV.
 *   Wq     : uint8 [N][K/2], low nibble = even k
 *   scales : fp16  [N][G], G = K/128
 *   zeros  : uint8 [N][(G+1)/2], two zero points per byte, low nibble = even group
 *   X      : bf16  [M][K]    Y : bf16 [M][N] (fp32 under the fp32 hook)
 *   Requires K % 128 == 0. `scales` needs only 2-byte alignment, `zeros` none.
 */
mbw_status gemv_int4_awq_g128(const uint8_t *Wq, const void *scales, const uint8_t *zeros,
                              const void *X, void *Y, int64_t M, int64_t N, int64_t K,
                              void *workspace, size_t ws_bytes, mbw_stream_t stream);

/*
 * mbw_repack_int4 -- the load-time reorder of INT4 codes (llm-rs vs vLLM,
 * sec. 6 "Quantization helps memory-bound work, and can hurt compute-bound
 * work": Marlin reorders 4-bit weights once at load time so that the unpack
 * hands each thread its operand directly; sec. 7 "Reading the scoreboard":
 * reordered weights and bit-trick unpacking). A row keeps its K/2 bytes.
 * Within each 4-byte word (codes of k = 8w .. 8w+7; nibble slot t = bits
 * 4t .. 4t+3 of the little-endian word, which holds k = 8w + t in the
 * canonical layout) code 8w + j moves to slot j/2 + 4*(j%2): the even k fill
 * slots 0-3 and the odd k slots 4-7, each in k order. The kernels' bit-trick
 * unpack (bits 0-3 with 16-19, then 4-7 with 20-23, ...) then yields the bf16
 * pairs (k0, k1), (k2, k3), ... in order, so they use X as loaded; with the
 * canonical layout they permute X on chip, per thread block. Applied three
 * times the reorder is the identity.
 *   Wq : uint8 [N][K/2], canonical (low nibble = even k)   Wr : uint8 [N][K/2]
 *   Requires K % 8 == 0; Wq and Wr 4-byte aligned; Wr may equal Wq (in place).
 */
mbw_status mbw_repack_int4(const uint8_t *Wq, uint8_t *Wr, int64_t N, int64_t K, mbw_stream_t stream);

/*
 * gemv_int4_awq_g128_repacked -- gemv_int4_awq_g128 with the codes in the
 * layout of mbw_repack_int4: same scales, zero points, X, Y and product (up to
 * the order of the fp32 additions). Same requirements as gemv_int4_awq_g128.
 * Its plans are keyed by MBW_OP_GEMV_INT4_AWQ_G128 | MBW_REPACKED and run on
 * the tensor-core kernel families (not the CUDA-core ones, which read the
 * canonical layout).
 */
mbw_status gemv_int4_awq_g128_repacked(const uint8_t *Wr, const void *scales, const uint8_t *zeros,
                                       const void *X, void *Y, int64_t M, int64_t N, int64_t K,
                                       void *workspace, size_t ws_bytes, mbw_stream_t stream);

/*
 * gemm_skinny_bf16 -- Y = X . W^T with BF16 weights and a skinny batch M
 * (tuned for 1 <= M <= 256; larger M is processed in slices of 256 rows).
 * The weights are still read once per call; at GB300's ridge (~286 FLOP per
 * byte) every M <= 256 stays memory-bound or near the ridge.
 *   X : bf16 [M][K]    W : bf16 [N][K]    Y : bf16 [M][N]
 *   Requires K % 8 == 0.
 */
mbw_status gemm_skinny_bf16(const void *X, const void *W, void *Y, int64_t M, int64_t N,
                            int64_t K, void *workspace, size_t ws_bytes, mbw_stream_t stream);

/*
 * gemv_int8_pc -- Y = X . W^T with symmetric INT8 weights and one fp32 scale
 * per output channel (TileInfer, "Pushing further with cheating: INT8
 * quantization"): w_ik = scales[i] * Wq[i][k], codes in [-127, 127]. The
 * kernel multiplies the codes in (exactly, as bf16 on the tensor core, fp32
 * accumulation) and applies the row's scale once to the finished sum. M = 1
 * is the decode GEMV; batches up to 8 run on the streaming GEMV kernels, and
 * batches above 8 on a batched mma.sync kernel that reads every weight once
 * per launch of 16, 32 or 64 rows.
 *   Wq     : int8 [N][K]     scales : fp32 [N]
 *   X      : bf16 [M][K]     Y      : bf16 [M][N] (fp32 under the fp32 hook)
 *   Requires K % 128 == 0. `scales` needs 4-byte alignment. The code -128 is
 *   outside the format; the kernels read it as -128.
 */
mbw_status gemv_int8_pc(const int8_t *Wq, const float *scales, const void *X, void *Y, int64_t M,
                        int64_t N, int64_t K, void *workspace, size_t ws_bytes, mbw_stream_t stream);

/*
 * mbw_quantize_int8_pc -- the load-time step that makes gemv_int8_pc's
 * weights from BF16 ones (same section): per row i, scales[i] = max_k |W[i][k]|
 * / 127 and Wq[i][k] = W[i][k] / scales[i] rounded to the nearest integer, so
 * the row's largest entry lands on +-127 and every entry is off by at most
 * half a scale. Both divisions are IEEE fp32; ties round to even; an all-zero
 * row gets scale 0 and codes 0. W must be finite.
 *   W : bf16 [N][K] (2-byte aligned)   Wq : int8 [N][K]   scales : fp32 [N]
 *   Any K >= 0.
 */
mbw_status mbw_quantize_int8_pc(const void *W, int8_t *Wq, float *scales, int64_t N, int64_t K,
                                mbw_stream_t stream);

/*
 * Optional fusions around one GEMV (all fields zero / NULL = none).
 *   norm_weight : bf16 [K] or NULL. RMSNorm prologue (llm-rs vs vLLM, "Decode:
 *                 from ~35% to ~70% of the ceiling": norms folded into the
 *                 projections): each batch row of X is replaced by
 *                 bf16(x * norm_weight / sqrt(mean(x^2) + norm_eps)) before the
 *                 product. Every CTA computes mean(x^2) over all of K itself
 *                 (fp32, fixed order), so the result is deterministic.
 *   norm_eps    : the epsilon under the square root.
 *   residual    : bf16 [M][N] or NULL. Residual epilogue (yalm, sec. 3.3:
 *                 matmul fused with add_residuals): Y = W.x + residual, rounded
 *                 once. It may be Y itself (in-place accumulation into the
 *                 residual stream).
 *   up_weights  : NULL, or a second weight matrix of the same format and shape
 *                 (with up_scales). Gated epilogue (yalm, sec. 3.3:
 *                 F.silu(w1(x)) * w3(x); TileInfer: SwiGLU in the GEMV
 *                 epilogue): Y = silu(W.x) * (U.x), silu(a) = a / (1 + e^-a),
 *                 both sums in fp32; the call streams both matrices. With a
 *                 residual too, the residual is added after the product.
 *   up_scales   : the up matrix's scales (INT4 g64: fp16 [N][K/64]; INT8:
 *                 fp32 [N]; AWQ: fp16 [N][K/128]; BF16: unused).
 *   up_zeros    : the up matrix's zero points (AWQ only: uint8 [N][(K/128+1)/2],
 *                 as gemv_int4_awq_g128's zeros); read by gemv_fused_awq_g128
 *                 alone, and only with up_weights set.
 */
typedef struct mbw_fusion {
    const void *norm_weight;
    float norm_eps;
    const void *residual;
    const void *up_weights;
    const void *up_scales;
    const void *up_zeros;
} mbw_fusion;

/*
 * gemv_fused -- one GEMV with the fusions of `fusion` (NULL: none), for
 * op = MBW_OP_GEMV_BF16, MBW_OP_GEMV_INT4_G64 (M = 1) or MBW_OP_GEMV_INT8_PC
 * (AWQ: gemv_fused_awq_g128, which also takes the zero points).
 * W / scales / X / Y and their layouts are those of the op's own call
 * (gemv_bf16: scales unused; gemv_int4_g64; gemv_int8_pc). Requires K > 0 and
 * the op's K multiple; norm_weight 16-byte aligned, up_weights 32-byte aligned,
 * residual 2-byte aligned. Y must not alias any input other than `residual`.
 * Fused calls run on the mma2 and latency kernel families; their plans are
 * keyed by op | MBW_FUSE_* (e.g. for mbw_autotune).
 */
mbw_status gemv_fused(int op, const void *W, const void *scales, const void *X, void *Y, int64_t M,
                      int64_t N, int64_t K, const mbw_fusion *fusion, void *workspace, size_t ws_bytes,
                      mbw_stream_t stream);

/*
 * gemv_fused_awq_g128 -- gemv_int4_awq_g128 (codes canonical, or in the
 * load-time repacked layout when `repacked` is 1) with the fusions of
 * `fusion` (NULL: none; the same prologue and epilogues as gemv_fused): the
 * RMSNorm prologue, the gated SiLU epilogue with an up matrix of the same
 * AWQ format (up_weights, up_scales, up_zeros; all three required together),
 * the residual add. Wq / scales / zeros / X / Y as in gemv_int4_awq_g128.
 * Requires K % 256 == 0 for a fused call (no fusion: K % 128 == 0); runs on
 * the streaming tensor-core kernel 4 batch rows per launch (larger batches in
 * slices of 4, each streaming the weights), whose smallest instantiation
 * needs K >= 1024 (MBW_ERR_UNSUPPORTED below it); plans keyed by
 * MBW_OP_GEMV_INT4_AWQ_G128 | MBW_FUSE_* (| MBW_REPACKED). Alignment as in
 * gemv_fused; up_zeros needs none.
 */
mbw_status gemv_fused_awq_g128(const uint8_t *Wq, const void *scales, const uint8_t *zeros, const void *X, void *Y,
                               int64_t M, int64_t N, int64_t K, int repacked, const mbw_fusion *fusion,
                               void *workspace, size_t ws_bytes, mbw_stream_t stream);

/* Bytes of workspace the largest plan of `op` may use for this shape (0 if none). */
size_t mbw_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * Dequantize INT4 weights to fp32 with the same unpack the GEMV kernels use:
 * out[i][k] = (q - 8) * s (g64) or (q - z) * s (AWQ). Both values are exact in
 * fp32 for every fp16 scale, so the result is bit-exact. Same layouts as above.
 */
mbw_status mbw_dequant_int4_g64(const uint8_t *Wq, const void *scales, float *out,
                                int64_t N, int64_t K, mbw_stream_t stream);
mbw_status mbw_dequant_int4_awq_g128(const uint8_t *Wq, const void *scales,
                                     const uint8_t *zeros, float *out, int64_t N,
                                     int64_t K, mbw_stream_t stream);

/* Test hook, per calling thread: 1 = later calls on this thread write fp32 y
 * (the fp32 accumulator before bf16 rounding), 0 = bf16 y (default). */
mbw_status mbw_set_output_fp32(int enable);

/*
 * Measure the candidate plans of (op, M, N, K) on `stream` and keep the
 * fastest (by achieved GB/s) in the plan cache. Blocking; allocates and frees
 * its own timing buffers; must not be called during stream capture.
 */
mbw_status mbw_autotune(int op, int64_t M, int64_t N, int64_t K, mbw_stream_t stream);

/* Number of candidate plans (kernel instantiation x split-K factor) valid
 * for (op, M, N, K); 0 for a bad op or shape. */
int mbw_plan_candidates(int op, int64_t M, int64_t N, int64_t K);

/* Make candidate `index` (0 .. mbw_plan_candidates()-1) the plan of this
 * shape, replacing the default or a tuned one. Lets a caller restore plans it
 * measured earlier, and lets tests run every kernel instantiation. */
mbw_status mbw_plan_select(int op, int64_t M, int64_t N, int64_t K, int index);

/* Index (among mbw_plan_candidates) of the plan this shape currently uses, so
 * that a tuned plan can be saved and restored with mbw_plan_select; -1 for a
 * bad op or shape. */
int mbw_plan_index(int op, int64_t M, int64_t N, int64_t K);

/* Write a one-line description of the plan a call of this shape would use
 * into buf (NUL-terminated, truncated to len). Returns MBW_OK. */
mbw_status mbw_plan_describe(int op, int64_t M, int64_t N, int64_t K, char *buf, size_t len);

/* Read and clear the device-side error flag set by bounded waits inside
 * kernels (synchronizes the current device). MBW_OK or MBW_ERR_DEVICE_TIMEOUT. */
mbw_status mbw_check_device_error(void);

/* Self-test of the failure path above. Launches two one-thread kernels on
 * `stream`, one per family of bounded waits (bulk-copy GEMV, tcgen05 GEMM);
 * each waits on a shared-memory mbarrier that nothing arrives at, gives up
 * after `tries` rounds (1 <= tries <= MBW_WAIT_LIMIT) and sets the fault flag
 * as a stalled kernel would. It touches no memory outside the kernels' own
 * shared memory and returns without synchronizing; the next
 * mbw_check_device_error() then reports MBW_ERR_DEVICE_TIMEOUT and clears the
 * flag. tries out of range: MBW_ERR_INVALID_ARG, nothing launched. */
mbw_status mbw_selftest_wait_expiry(int64_t tries, mbw_stream_t stream);

/* Host-side fault injection (test hook). The next `count` calls on the
 * calling thread that pass their argument checks and would launch a kernel
 * (the GEMV/GEMM entry points, mbw_repack_int4, mbw_quantize_int8_pc and the
 * dequant helpers) launch nothing and return MBW_ERR_CUDA, as a failed launch
 * would, with mbw_last_error() naming the injection. count = 0 (the default)
 * turns it off; a negative count is MBW_ERR_INVALID_ARG. */
mbw_status mbw_inject_launch_failures(int count);

/* Number of kernel launches this library has issued on the calling thread. */
uint64_t mbw_launch_count(void);

const char *mbw_status_string(mbw_status status);
/* Detail of the last failed call on the calling thread ("" if none). */
const char *mbw_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MBW_H */
