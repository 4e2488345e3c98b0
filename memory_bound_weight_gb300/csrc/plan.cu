// plan.cu -- launch-time plan selection for the streaming GEMV kernels.
//
// A plan is (kernel family, instantiation, split-K cluster size, k-slices per
// CTA). The default plan is a heuristic; mbw_autotune() replaces it by
// measurement, in the manner of tinyinfer's load-time autotuner ("R rows per
// warp" section: time R = 1, 2, 4 on every distinct matrix shape at model load
// and keep the fastest, in a few milliseconds). Here the candidates are every
// instantiation of both kernel families x split {1, 2, 4, 8} (x k-slices per
// CTA for the tensor-core family); each is timed as a CUDA graph of
// back-to-back launches over rotating weight copies larger than L2 (the
// regime a matrix sees inside a decode step), and the highest GB/s wins.
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "internal.h"
#include "mbw.h"

namespace mbw {

static std::mutex g_plan_mu;
static std::map<std::tuple<int, int, int64_t, int64_t, int64_t>, Plan> g_plans;

static const size_t kSmemLimit = kSmemFit;

static int fmt_of_op(int op) {
    switch (op & MBW_OP_BASE_MASK) {
        case MBW_OP_GEMV_INT4_G64: return FMT_G64;
        case MBW_OP_GEMV_INT4_AWQ_G128: return FMT_AWQ;
        case MBW_OP_GEMV_INT8_PC: return FMT_I8;
        default: return FMT_BF16;
    }
}

static int chunks_of(int fmt, int64_t K) { return (int)(fmt == FMT_BF16 ? K / 8 : fmt == FMT_I8 ? K / 16 : K / 32); }

static size_t simt_smem(int fmt, const SimtConfig& c, int64_t K, int split) {
    GemvArgs a{};
    a.chunks = chunks_of(fmt, K);
    a.split_chunks = (a.chunks + split - 1) / split;
    return simt_smem_bytes(fmt, c, a, split);
}

// SIMT batch width for a call of M rows: the smallest kernel batch >= min(M, 8).
static int simt_want_mb(int64_t M) { return M <= 2 ? (int)M : M <= 4 ? 4 : 8; }

// n-blocks of 8 columns the batched AWQ mma.sync kernel runs for a call of M
// rows: the fewest covering min(M, 64).
static int awqb_want_nb(int64_t M) {
    const int64_t m = std::min<int64_t>(M, 64);
    return m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8;
}

// Plan-cache key of the batch: calls whose M share a key share a plan, so
// every candidate valid for one M of a key must be valid for all of them.
static int batch_key(int op, int64_t M) {
    if (op == MBW_OP_GEMM_SKINNY_BF16 && M > 8) return tc_batch_tile(M);
    if ((op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT4_AWQ_G128 && M > 4) return 1000 + 8 * awqb_want_nb(M);
    if ((op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT8_PC && M > 8) return 1000 + 8 * awqb_want_nb(M);
    return (int)std::min<int64_t>(M, 8);
}

int plan_batch_width(int fmt, const Plan& p) {
    if (p.kind == PLAN_TC) return 1 << 30;  // one launch covers the whole batch
    if (p.kind == PLAN_AWQB) return 8 * awqb_config(p.cfg).nb;
    if (p.kind == PLAN_MMA2) return mma2_max_batch(fmt);
    if (p.kind == PLAN_LAT) return lat_max_batch(fmt);
    if (p.kind == PLAN_MMA || p.kind == PLAN_TMA) return mma_max_batch(fmt);
    if (p.kind == PLAN_ROWS) return 1;
    if (p.kind == PLAN_QBULK) return mma2_max_batch(fmt);
    return simt_config(fmt, p.cfg).mb;
}

static int64_t kblocks(int fmt, int64_t K) {
    const int BK = (fmt == FMT_BF16) ? 32 : 128;
    return (K + BK - 1) / BK;
}

// `flags`: the MBW_FUSE_* and MBW_REPACKED bits of the call. Repacked INT4
// codes run on every pair-based tensor-core kernel (they stage x as loaded);
// the SIMT kernels read canonical codes. Fused calls run on the "mma2" and
// latency families only (the kernels with the prologue and epilogue hooks).
static bool plan_valid(int fmt, const Plan& p, int64_t M, int64_t N, int64_t K, int flags = 0) {
    const int fuse = flags & MBW_FUSE_MASK;
    if ((flags & MBW_REPACKED) && p.kind == PLAN_SIMT) return false;
    if (p.split < 1 || p.split > 8) return false;
    const int glu = (fuse & MBW_FUSE_GLU) ? 1 : 0;
    if (fuse && p.kind != PLAN_MMA2 && p.kind != PLAN_LAT) return false;
    if (p.kind == PLAN_TC) {
        // tensor-core skinny GEMM: BF16, batches above the GEMV column width
        if (fmt == FMT_AWQ) {
            // AWQ tensor-core GEMM: batches above the GEMV column width, one 128-k group per stage
            const int64_t G = K / 128;
            if (M <= 4 || K % 128 != 0 || p.cfg != 0 || p.occ != 1 || p.split > G) return false;
            const int64_t per = ((G + p.split - 1) / p.split + 3) / 4 * 4;  // whole 4-group ring slots per rank
            return per * (p.split - 1) < G && tc_awq_fits(M, K, p.split);
        }
        // cfg bit 0: ring (deep / co-resident), bit 1: two 64-k boxes per stage, bit 2: CTA pairs
        // (batches 5 .. 8 run in a 16-wide tile: the tensor-core kernel can still beat the GEMVs)
        if (fmt != FMT_BF16 || M <= 4 || p.cfg < 0 || p.cfg > 7 || p.occ != 1) return false;
        if ((p.cfg & 4) && (tc_batch_tile(M) < 128 || p.split > 4)) return false;
        const int64_t bk = (p.cfg & 2) ? 128 : 64;
        const int64_t KS = (K + bk - 1) / bk;
        if (p.split > KS) return false;
        const int64_t per = (KS + p.split - 1) / p.split;
        return per * (p.split - 1) < KS;  // every cluster rank gets k-stages
    }
    if (p.kind == PLAN_AWQB) {
        // batched AWQ on mma.sync: batches above the GEMV column width, whole
        // super-blocks of 256 k, at least one per cluster rank
        // (INT8: batches above the INT8 GEMVs' 8 rows, whole 128-k super-blocks)
        if ((fmt != FMT_AWQ && fmt != FMT_I8) || p.cfg < 0 || p.cfg >= awqb_num_configs()) return false;
        if (M <= (fmt == FMT_I8 ? 8 : 4)) return false;
        const AwqbConfig c = awqb_config(p.cfg);
        if (c.fmt != fmt) return false;
        const int64_t bks = (fmt == FMT_I8) ? 128 : 256;
        // the fewest n-blocks covering the batch, or down to a quarter of them
        // in slices (each slice streams the weights again; past 16 rows the
        // kernel is bound by the MMA rate rather than the weight stream, and
        // narrower slices stage less of X in shared memory)
        const int want = awqb_want_nb(M);
        if (c.nb > want || 4 * c.nb < want) return false;
        if (K % bks != 0 || p.occ < 1 || p.occ > c.minb || K / bks < p.split) return false;
        if ((uint64_t)N * (uint64_t)(fmt == FMT_I8 ? K : K / 2) > 0xFFFFFFFFull) return false;  // 32-bit offsets
        const size_t sm = awqb_smem_bytes(c, N, K, p.split, p.occ);
        return sm <= kSmemLimit && sm * p.occ <= (size_t)227 * 1024;
    }
    if (p.kind == PLAN_SIMT) {
        if (p.cfg < 0 || p.cfg >= simt_num_configs(fmt)) return false;
        const SimtConfig c = simt_config(fmt, p.cfg);
        if (c.persist) {
            // occ CTAs per SM, each holding the whole of x; at least one row group per warp
            if (M != 1 || p.split != 1 || p.occ < 1 || p.occ * c.warps > 32 || K % 16 != 0) return false;
            if ((int64_t)device_sm_count() * p.occ * c.warps * c.r > N) return false;
            return simt_smem(fmt, c, K, 1) * p.occ <= (size_t)227 * 1024;
        }
        if (p.occ != 1) return false;
        if (c.mb != simt_want_mb(M)) return false;
        if (c.cb == 32 && (fmt != FMT_BF16 || K % 16 != 0)) return false;  // whole 32-byte chunks per row
        if (simt_smem(fmt, c, K, p.split) > kSmemLimit) return false;
        const int chunks = chunks_of(fmt, K) / (c.cb / 16);
        if (p.split > 1 && (chunks + p.split - 1) / p.split < 16) return false;
        return true;
    }
    if (p.kind == PLAN_MMA) {
        if (p.cfg < 0 || p.cfg >= mma_num_configs(fmt)) return false;
        const MmaConfig c = mma_config(fmt, p.cfg);
        if (p.occ < 1 || p.occ > 2) return false;
        const int mb = (int)std::min<int64_t>(M, mma_max_batch(fmt));
        // whole row blocks only, and every warp of the cluster gets at least one
        if (K % (fmt == FMT_BF16 ? 32 : 128) != 0) return false;
        if ((int64_t)p.split * c.warps > kblocks(fmt, K)) return false;
        if (mma_smem_bytes(fmt, c, N, K, mb, p.split, p.occ) > kSmemLimit) return false;
        return true;
    }
    if (p.kind == PLAN_MMA2) {
        if (p.cfg < 0 || p.cfg >= mma2_num_configs(fmt)) return false;
        const MmaConfig c = mma2_config(fmt, p.cfg);
        if (p.occ < 1 || p.occ > 2) return false;
        const int bk = mma2_block_k(fmt);
        if (K % bk != 0) return false;
        const int mb = (int)std::min<int64_t>(M, mma2_max_batch(fmt));
        if ((int64_t)p.split * c.warps > K / bk) return false;
        if (mma2_smem_bytes(fmt, c, N, K, mb, p.split, p.occ, glu) > kSmemLimit) return false;
        return true;
    }
    if (p.kind == PLAN_LAT) {
        if (p.cfg < 0 || p.cfg >= lat_num_configs(fmt)) return false;
        const LatConfig c = lat_config(fmt, p.cfg);
        if (p.occ < 1 || p.occ > 2) return false;
        const int mb = (int)std::min<int64_t>(M, lat_max_batch(fmt));
        const int items = lat_items_per_warp(fmt, c, N, K, p.split, p.occ, glu);
        if (items < 1 || items > c.ni) return false;
        if (c.ni > items + 1) return false;  // a smaller instantiation holds this share
        if (lat_smem_bytes(fmt, c, N, K, mb, p.split, p.occ, glu, fuse ? 1 : 0) > kSmemLimit) return false;
        return true;
    }
    if (p.kind == PLAN_QBULK) {
        // INT4 (group-64, AWQ) and INT8 at the "mma2" batch widths, whole 128-byte super-blocks, no fusions
        if ((fmt != FMT_G64 && fmt != FMT_AWQ && fmt != FMT_I8) || p.cfg < 0 || p.cfg >= qbulk_num_configs(fmt))
            return false;
        const int64_t bk = (fmt == FMT_I8) ? 128 : 256;
        if (M > mma2_max_batch(fmt) || K % bk != 0 || p.occ < 1 || p.occ > 2 || K / bk < p.split) return false;
        const size_t sm = qbulk_smem_bytes(fmt, qbulk_config(fmt, p.cfg), N, K, (int)M, p.split, p.occ);
        return sm * p.occ <= (size_t)227 * 1024;
    }
    if (p.kind == PLAN_ROWS) {
        // BF16 batch 1, one CTA row range per SM (or two), x staged whole
        if (fmt != FMT_BF16 || M != 1 || p.split != 1 || p.cfg < 0 || p.cfg >= rows_num_configs()) return false;
        if (p.occ < 1 || p.occ > 2 || 2 * K > 64 * 1024) return false;
        const size_t sm = rows_smem_bytes(rows_config(p.cfg), N, K, p.occ);
        return sm <= (size_t)227 * 1024 / p.occ && (p.occ == 1 || sm <= kSmemLimit);
    }
    if (p.kind == PLAN_TMA) {
        if (p.cfg < 0 || p.cfg >= tma_num_configs(fmt)) return false;
        const TmaConfig c = tma_config(fmt, p.cfg);
        if (p.occ < 1 || p.occ > 2) return false;
        const int mb = (int)std::min<int64_t>(M, mma_max_batch(fmt));
        if (K % (fmt == FMT_BF16 ? 32 : 128) != 0) return false;
        if ((int64_t)p.split > kblocks(fmt, K)) return false;
        if (tma_smem_bytes(fmt, c, N, K, mb, p.split, p.occ) > kSmemLimit) return false;
        return true;
    }
    return false;
}

static std::vector<Plan> candidates(int op, int64_t M, int64_t N, int64_t K) {
    std::vector<Plan> out;
    const int fmt = fmt_of_op(op);
    const int flags = op & (MBW_FUSE_MASK | MBW_REPACKED);
    const int64_t Mb = std::min<int64_t>(M, 8);
    if ((op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT4_AWQ_G128 && M > 4) {
        for (int sp = 1; sp <= 8; ++sp) {
            Plan p{PLAN_TC, 0, sp, 1};
            if (plan_valid(fmt, p, M, N, K, flags)) out.push_back(p);
        }
        for (int cfg = 0; cfg < awqb_num_configs(); ++cfg)
            for (int sp = 1; sp <= 8; sp *= 2)
                for (int occ = 1; occ <= 2; ++occ) {
                    Plan p{PLAN_AWQB, cfg, sp, occ};
                    if (plan_valid(fmt, p, M, N, K, flags)) out.push_back(p);
                }
    }
    if ((op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT8_PC && M > 8)
        for (int cfg = 0; cfg < awqb_num_configs(); ++cfg)
            for (int sp = 1; sp <= 8; sp *= 2)
                for (int occ = 1; occ <= 2; ++occ) {
                    Plan p{PLAN_AWQB, cfg, sp, occ};
                    if (plan_valid(fmt, p, M, N, K, flags)) out.push_back(p);
                }
    if (op == MBW_OP_GEMM_SKINNY_BF16 && M > 4)
        for (int cfg = 0; cfg <= 7; ++cfg)
            for (int sp = 1; sp <= 8; ++sp) {
                Plan p{PLAN_TC, cfg, sp, 1};
                if (plan_valid(fmt, p, M, N, K, flags)) out.push_back(p);
            }
    const int splits[4] = {1, 2, 4, 8};
    for (int cfg = 0; cfg < mma_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 2; ++occ) {
                Plan p{PLAN_MMA, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    for (int cfg = 0; cfg < mma2_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 2; ++occ) {
                Plan p{PLAN_MMA2, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    for (int cfg = 0; cfg < lat_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 2; ++occ) {
                Plan p{PLAN_LAT, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    for (int cfg = 0; cfg < qbulk_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 2; ++occ) {
                Plan p{PLAN_QBULK, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    for (int cfg = 0; cfg < rows_num_configs(); ++cfg)
        for (int occ = 1; occ <= 2; ++occ) {
            Plan p{PLAN_ROWS, cfg, 1, occ};
            if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
        }
    for (int cfg = 0; cfg < tma_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 2; ++occ) {
                Plan p{PLAN_TMA, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    for (int cfg = 0; cfg < simt_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si)
            for (int occ = 1; occ <= 8; ++occ) {
                Plan p{PLAN_SIMT, cfg, splits[si], occ};
                if (plan_valid(fmt, p, Mb, N, K, flags)) out.push_back(p);
            }
    return out;
}

static Plan plan_heuristic(int op, int64_t M, int64_t N, int64_t K) {
    const int fmt = fmt_of_op(op);
    const int flags = op & (MBW_FUSE_MASK | MBW_REPACKED);
    const int fuse = op & MBW_FUSE_MASK;
    const int64_t Mb = std::min<int64_t>(M, 8);
    const int sms = device_sm_count();
    const bool awq_batch = (op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT4_AWQ_G128 && M > 4;
    const bool i8_batch = (op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT8_PC && M > 8 && !fuse;
    if (awq_batch || i8_batch) {
        // batched AWQ / INT8 on mma.sync: 8 warps; split K over a cluster
        // while the 16-row tiles do not cover the SMs or X does not fit
        const int want = awqb_want_nb(M);
        const int bks = i8_batch ? 128 : 256;
        for (int i = 0; i < awqb_num_configs(); ++i) {
            const AwqbConfig c = awqb_config(i);
            if (c.fmt != fmt || c.nb != want || c.wt * c.wk != 8) continue;
            const int64_t tiles = (N + 15) / 16;
            for (int occ = c.minb; occ >= 1; --occ) {
                // split while the tiles do not cover the SMs or X does not fit
                Plan p{PLAN_AWQB, i, 1, occ};
                while (p.split < 8 && K / bks / (2 * p.split) >= c.wk &&
                       (tiles * p.split < (int64_t)sms * occ || !plan_valid(fmt, p, M, N, K, flags)))
                    p.split *= 2;
                if (plan_valid(fmt, p, M, N, K, flags)) return p;
            }
            break;
        }
    }
    if ((op == MBW_OP_GEMM_SKINNY_BF16 && M > 8) ||
        ((op & MBW_OP_BASE_MASK) == MBW_OP_GEMV_INT4_AWQ_G128 && M > 4)) {
        // tcgen05 tiles of 128 weight rows; split K over a cluster until the
        // tiles cover the SMs
        const int64_t tiles = (N + 127) / 128;
        int split = 1;
        while (split < 8 && tiles * (split + 1) <= sms) ++split;
        Plan p{PLAN_TC, 0, split, 1};
        while (!plan_valid(fmt, p, M, N, K, flags) && p.split > 1) --p.split;
        return p;
    }
    if (fmt == FMT_I8 || fuse) {
        // INT8 and fused calls run on the "mma2" and latency families only: 8
        // warps, 3 super-blocks in flight in registers, one CTA per SM; split K
        // over a cluster while there are fewer 16-row tiles than SMs.
        const int64_t tiles = (N + 15) / 16;
        Plan p{PLAN_MMA2, 1, 1, 1};
        while (p.split < 8 && tiles * p.split < sms && (int64_t)8 * p.split * 2 <= K / 128) p.split *= 2;
        while (!plan_valid(fmt, p, Mb, N, K, flags) && p.split > 1) p.split /= 2;
        if (plan_valid(fmt, p, Mb, N, K, flags)) return p;
        const std::vector<Plan> c = candidates(op, M, N, K);
        if (!c.empty()) return c.front();
        return p;
    }
    // Tensor-core family: 8 warps, 4 blocks in flight, one CTA per SM; split K
    // over a cluster while there are fewer 16-row tiles than SMs.
    int cfg = 0;
    for (int i = 0; i < mma_num_configs(fmt); ++i) {
        const MmaConfig c = mma_config(fmt, i);
        if (c.warps == 8 && c.u == 4) {
            cfg = i;
            break;
        }
    }
    const int64_t tiles = (N + 15) / 16;
    const int64_t KB = kblocks(fmt, K);
    int split = 1;
    while (split < 8 && tiles * split < sms && (int64_t)8 * split * 2 <= KB) split *= 2;
    Plan p{PLAN_MMA, cfg, split, 1};
    while (!plan_valid(fmt, p, Mb, N, K, flags) && p.split < 8) p.split *= 2;
    if (plan_valid(fmt, p, Mb, N, K, flags)) return p;
    const std::vector<Plan> c = candidates(op, M, N, K);
    if (!c.empty()) return c.front();
    return Plan{PLAN_MMA, cfg, 8, 1};
}

// The built-in plan of a shape: the heuristic's pick when it is one of the
// shape's candidates, else the first candidate, else PLAN_NONE (no kernel
// fits: x of one CTA's k-range, even split over the largest cluster, does not
// fit shared memory).
Plan plan_default(int op, int64_t M, int64_t N, int64_t K) {
    const Plan h = plan_heuristic(op, M, N, K);
    const std::vector<Plan> c = candidates(op, M, N, K);
    for (const Plan& p : c)
        if (p.kind == h.kind && p.cfg == h.cfg && p.split == h.split && p.occ == h.occ) return h;
    if (!c.empty()) return c.front();
    return Plan{PLAN_NONE, 0, 1, 1};
}

static int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

static std::tuple<int, int, int64_t, int64_t, int64_t> key_of(int op, int64_t M, int64_t N, int64_t K) {
    return std::make_tuple(current_device(), op, (int64_t)batch_key(op, M), N, K);
}

Plan plan_lookup(int op, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    (void)s;
    const auto key = key_of(op, M, N, K);
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) return it->second;
    }
    const Plan p = plan_default(op, M, N, K);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans.emplace(key, p);
    return p;
}

std::string plan_to_string(int op, const Plan& p) {
    if (p.kind == PLAN_NONE) return "none (no kernel fits this shape)";
    const int fmt = fmt_of_op(op);
    const char* fs = fmt == FMT_BF16 ? "bf16" : fmt == FMT_G64 ? "int4_g64" : fmt == FMT_I8 ? "int8_pc" : "int4_awq_g128";
    char buf[192];
    if (p.kind == PLAN_AWQB) {
        const AwqbConfig c = awqb_config(p.cfg);
        snprintf(buf, sizeof(buf),
                 "%s fmt=%s batch_cols=%d warps=%d (tiles %d x k %d) superblocks_in_flight=%d ring=%s "
                 "ctas_per_sm=%d split_k=%d",
                 c.fmt == FMT_I8 ? "int8_mma" : "awq_mma", fs, 8 * c.nb, c.wt * c.wk, c.wt, c.wk, c.u,
                 c.async ? "smem" : c.early ? "registers refill=early" : "registers refill=late", p.occ, p.split);
    } else if (p.kind == PLAN_TC) {
        if (fmt == FMT_AWQ)
            snprintf(buf, sizeof(buf), "tcgen05 fmt=%s tile=128xbatch k_stage=128 (one group) split_k=%d", fs, p.split);
        else
            snprintf(buf, sizeof(buf), "tcgen05 fmt=%s tile=%sxbatch k_stage=%d ring=%s split_k=%d", fs,
                     (p.cfg & 4) ? "256 (cta pair)" : "128", (p.cfg & 2) ? 128 : 64,
                     (p.cfg & 1) ? "shared_sm" : "deep", p.split);
    } else if (p.kind == PLAN_LAT) {
        const LatConfig c = lat_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf),
                 "lat fmt=%s warps=%d (k %d x tiles %d) items_per_warp<=%d unpacked_before_wait=%d staging=%s%s "
                 "ctas_per_sm=%d split_k=%d",
                 fs, c.warps, c.warps / c.wt, c.wt, c.ni, c.npre, c.staged ? "smem" : "registers",
                 c.lean ? " lean" : "", p.occ, p.split);
    } else if (p.kind == PLAN_MMA2) {
        const MmaConfig c = mma2_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf), "mma2 fmt=%s warps=%d superblocks_in_flight=%d ring=%s ctas_per_sm=%d split_k=%d",
                 fs, c.warps, c.u, c.async ? "cp.async" : "registers", p.occ, p.split);
    } else if (p.kind == PLAN_TMA) {
        const TmaConfig c = tma_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf), "tma fmt=%s consumer_warps=%d ring_stages=%d ctas_per_sm=%d split_k=%d", fs,
                 c.warps, c.depth, p.occ, p.split);
    } else if (p.kind == PLAN_QBULK) {
        const QbulkConfig c = qbulk_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf),
                 "bulk fmt=%s consumer_warps=%d ring_stages=%d superblocks_per_warp=%d ctas_per_sm=%d split_k=%d", fs,
                 c.warps, c.depth, c.bsc, p.occ, p.split);
    } else if (p.kind == PLAN_ROWS) {
        const RowsConfig c = rows_config(p.cfg);
        snprintf(buf, sizeof(buf), "rows fmt=%s warps=%d ring_slots_per_warp=%d stage_bytes=%d ctas_per_sm=%d split_k=%d",
                 fs, c.warps, c.depth, c.seg, p.occ, p.split);
    } else if (p.kind == PLAN_MMA) {
        const MmaConfig c = mma_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf), "mma fmt=%s warps=%d blocks_in_flight=%d ctas_per_sm=%d split_k=%d", fs, c.warps,
                 c.u, p.occ, p.split);
    } else {
        const SimtConfig c = simt_config(fmt, p.cfg);
        snprintf(buf, sizeof(buf),
                 "simt fmt=%s warps=%d rows_per_warp=%d chunks_in_flight=%d chunk_bytes=%d batch=%d split_k=%d%s", fs,
                 c.warps, c.r, c.u, c.cb, c.mb, p.split,
                 c.persist ? (" persistent ctas_per_sm=" + std::to_string(p.occ)).c_str() : "");
    }
    std::string out = buf;
    if (op & MBW_FUSE_NORM) out += " +rmsnorm";
    if (op & MBW_FUSE_GLU) out += " +swiglu";
    if (op & MBW_FUSE_RESIDUAL) out += " +residual";
    if (op & MBW_REPACKED) out += " codes=repacked";
    return out;
}

cudaError_t launch_plan(int fmt, const Plan& p, const GemvArgs& a, cudaStream_t s) {
    if (p.kind == PLAN_AWQB) return launch_gemv_awq_batch(p, a, s);
    if (p.kind == PLAN_TC && fmt == FMT_AWQ)
        return launch_gemm_tc_awq(a.W, a.scales, a.zeros, a.x, a.y, a.M, a.N, a.K, p.split, a.out_f32, a.x_natural,
                                  s);
    if (p.kind == PLAN_TC) return launch_gemm_tc(a.x, (const uint16_t*)a.W, a.y, a.M, a.N, a.K, p.split, p.cfg, a.out_f32, s);
    if (p.kind == PLAN_MMA2) return launch_gemv_mma2(fmt, p, a, s);
    if (p.kind == PLAN_LAT) return launch_gemv_lat(fmt, p, a, s);
    if (p.kind == PLAN_TMA) return launch_gemv_tma(fmt, p, a, s);
    if (p.kind == PLAN_ROWS) return launch_gemv_rows(p, a, s);
    if (p.kind == PLAN_QBULK) return launch_gemv_qbulk(fmt, p, a, s);
    if (p.kind == PLAN_MMA) return launch_gemv_mma(fmt, p, a, s);
    return launch_gemv_simt(fmt, p, a, s);
}

static size_t weight_bytes(int fmt, int64_t N, int64_t K) {
    if (fmt == FMT_BF16) return (size_t)N * K * 2;
    if (fmt == FMT_G64) return (size_t)N * K / 2 + (size_t)N * (K / 64) * 2;
    if (fmt == FMT_I8) return (size_t)N * K + (size_t)N * 4;
    const int64_t G = K / 128;
    return (size_t)N * K / 2 + (size_t)N * G * 2 + (size_t)N * ((G + 1) / 2);
}

static bool shape_ok(int op, int64_t M, int64_t N, int64_t K) {
    const int base = op & MBW_OP_BASE_MASK, flags = op & ~MBW_OP_BASE_MASK;
    if (base < MBW_OP_GEMV_BF16 || base > MBW_OP_GEMV_INT8_PC) return false;
    if (flags & ~(MBW_FUSE_MASK | MBW_REPACKED)) return false;
    const int fuse = flags & MBW_FUSE_MASK;
    if ((flags & MBW_REPACKED) && base != MBW_OP_GEMV_INT4_AWQ_G128) return false;
    if (fuse && base == MBW_OP_GEMM_SKINNY_BF16) return false;
    if (M < 1 || N < 1 || K < 1 || N > MBW_MAX_DIM || K > MBW_MAX_DIM || M > MBW_MAX_DIM) return false;
    if (base == MBW_OP_GEMV_INT4_G64 && M != 1) return false;
    const int fmt = fmt_of_op(op);
    const int64_t kunit = fmt == FMT_BF16 ? 8 : fmt == FMT_G64 ? 64 : 128;  // AWQ and INT8: 128
    return K % kunit == 0;
}

}  // namespace mbw

using namespace mbw;

extern "C" mbw_status mbw_plan_describe(int op, int64_t M, int64_t N, int64_t K, char* buf, size_t len) {
    if (!buf || len == 0) return MBW_ERR_INVALID_ARG;
    if (!shape_ok(op, M, N, K)) {
        set_last_error("mbw_plan_describe: bad op or shape");
        return MBW_ERR_INVALID_ARG;
    }
    const Plan p = plan_lookup(op, M, N, K, nullptr);
    snprintf(buf, len, "%s", plan_to_string(op, p).c_str());
    return MBW_OK;
}

extern "C" int mbw_plan_candidates(int op, int64_t M, int64_t N, int64_t K) {
    if (!shape_ok(op, M, N, K)) return 0;
    return (int)candidates(op, M, N, K).size();
}

extern "C" int mbw_plan_index(int op, int64_t M, int64_t N, int64_t K) {
    if (!shape_ok(op, M, N, K)) return -1;
    const Plan cur = plan_lookup(op, M, N, K, nullptr);
    const std::vector<Plan> c = candidates(op, M, N, K);
    for (size_t i = 0; i < c.size(); ++i)
        if (c[i].kind == cur.kind && c[i].cfg == cur.cfg && c[i].split == cur.split && c[i].occ == cur.occ)
            return (int)i;
    return -1;
}

extern "C" mbw_status mbw_plan_select(int op, int64_t M, int64_t N, int64_t K, int index) {
    if (!shape_ok(op, M, N, K)) {
        set_last_error("mbw_plan_select: bad op or shape");
        return MBW_ERR_INVALID_ARG;
    }
    const std::vector<Plan> c = candidates(op, M, N, K);
    if (index < 0 || index >= (int)c.size()) {
        set_last_error("mbw_plan_select: index out of range");
        return MBW_ERR_INVALID_ARG;
    }
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[key_of(op, M, N, K)] = c[index];
    return MBW_OK;
}

extern "C" mbw_status mbw_autotune(int op, int64_t M, int64_t N, int64_t K, mbw_stream_t stream_) {
    cudaStream_t user = (cudaStream_t)stream_;
    if (!shape_ok(op, M, N, K)) {
        set_last_error("mbw_autotune: bad op or shape");
        return MBW_ERR_INVALID_ARG;
    }
    cudaStreamCaptureStatus cs;
    if (cudaStreamIsCapturing(user, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) {
        set_last_error("mbw_autotune: stream is capturing");
        return MBW_ERR_INVALID_ARG;
    }
    // Timing graphs are captured on a private stream (the caller's may be the
    // legacy default stream, which cannot be captured); the caller's stream is
    // drained first so that tuning does not overlap its work.
    cudaError_t e = cudaStreamSynchronize(user);
    cudaStream_t stream = nullptr;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        set_last_error(std::string("mbw_autotune: ") + cudaGetErrorString(e));
        return MBW_ERR_CUDA;
    }
    const int fmt = fmt_of_op(op);
    // candidates are timed at the call's batch (a GEMV plan narrower than M
    // is launched once per batch slice, as the call would)
    const int64_t Mb = M;
    const int fuse = op & MBW_FUSE_MASK;
    const int glu = (fuse & MBW_FUSE_GLU) ? 1 : 0;
    const size_t wb1 = weight_bytes(fmt, N, K);
    const size_t wstride1 = (wb1 + 255) / 256 * 256;
    const size_t wb = glu ? 2 * wstride1 : wb1;  // gated calls stream the gate and the up matrix
    const size_t wstride = (wb + 255) / 256 * 256;
    const size_t target = (size_t)384 << 20;  // about three times the L2
    int copies = (int)std::max<size_t>(2, (target + wb - 1) / wb);
    copies = std::min(copies, 96);
    const int launches = copies;  // one launch per copy: the first launch's ramp counts, as after a shape change

    uint8_t* wbuf = nullptr;
    uint16_t* xbuf = nullptr;
    void* ybuf = nullptr;
    uint16_t* nbuf = nullptr;  // RMSNorm weight
    uint16_t* rbuf = nullptr;  // residual
    e = cudaMalloc(&wbuf, wstride * copies);
    if (e == cudaSuccess) e = cudaMalloc(&xbuf, (size_t)Mb * K * 2);
    if (e == cudaSuccess) e = cudaMalloc(&ybuf, (size_t)Mb * N * 4);
    if (e == cudaSuccess && (fuse & MBW_FUSE_NORM)) e = cudaMalloc(&nbuf, (size_t)K * 2);
    if (e == cudaSuccess && (fuse & MBW_FUSE_RESIDUAL)) e = cudaMalloc(&rbuf, (size_t)Mb * N * 2);
    if (e == cudaSuccess) e = cudaMemsetAsync(wbuf, 0x37, wstride * copies, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(xbuf, 0x37, (size_t)Mb * K * 2, stream);
    if (e == cudaSuccess && nbuf) e = cudaMemsetAsync(nbuf, 0x37, (size_t)K * 2, stream);
    if (e == cudaSuccess && rbuf) e = cudaMemsetAsync(rbuf, 0x37, (size_t)Mb * N * 2, stream);
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    if (e == cudaSuccess) e = cudaEventCreate(&t0);
    if (e == cudaSuccess) e = cudaEventCreate(&t1);

    Plan best = plan_default(op, M, N, K);
    float best_ms = 1e30f;
    const std::vector<Plan> cands = candidates(op, M, N, K);
    for (size_t ci = 0; ci < cands.size() && e == cudaSuccess; ++ci) {
        const Plan p = cands[ci];
        GemvArgs a{};
        a.N = (int)N;
        a.K = (int)K;
        a.M = (int)std::min<int64_t>(Mb, (int64_t)plan_batch_width(fmt, p));
        a.x = xbuf;
        a.y = ybuf;
        a.chunks = chunks_of(fmt, K);
        a.split_chunks = (a.chunks + p.split - 1) / p.split;
        a.groups = (int)(fmt == FMT_G64 ? K / 64 : fmt == FMT_AWQ ? K / 128 : 0);
        a.zstride = (a.groups + 1) / 2;
        a.out_f32 = 0;
        a.norm_w = nbuf;
        a.norm_eps = 1e-6f;
        a.residual = rbuf;
        a.glu = glu;
        a.x_natural = (op & MBW_REPACKED) ? 1 : 0;
        const size_t codes = fmt == FMT_BF16 ? (size_t)N * K * 2 : fmt == FMT_I8 ? (size_t)N * K : (size_t)N * K / 2;
        const int slices = (int)((Mb + a.M - 1) / a.M);  // launches per call at this batch
        cudaGraph_t g = nullptr;
        cudaGraphExec_t ge = nullptr;
        e = cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) break;
        cudaError_t le = cudaSuccess;
        for (int i = 0; i < launches && le == cudaSuccess; ++i) {
            a.W = wbuf + (size_t)(i % copies) * wstride;
            a.scales = (const uint16_t*)(a.W + codes);
            a.zeros = (const uint8_t*)(a.W + codes + (size_t)N * a.groups * 2);
            a.rscale = (const float*)(a.W + codes);
            if (glu) {
                a.W2 = a.W + wstride1;
                a.scales2 = (const uint16_t*)(a.W2 + codes);
                a.rscale2 = (const float*)(a.W2 + codes);
                a.zeros2 = (const uint8_t*)(a.W2 + codes + (size_t)N * a.groups * 2);
            }
            for (int sl = 0; sl < slices && le == cudaSuccess; ++sl) le = launch_plan(fmt, p, a, stream);
        }
        e = cudaStreamEndCapture(stream, &g);
        if (le != cudaSuccess || e != cudaSuccess) {
            // a candidate that cannot launch here (e.g. a cluster shape the
            // device cannot schedule) is skipped
            if (g) cudaGraphDestroy(g);
            cudaGetLastError();
            e = cudaSuccess;
            continue;
        }
        e = cudaGraphInstantiate(&ge, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) {
            cudaGetLastError();
            e = cudaSuccess;
            continue;
        }
        float times[3] = {0.f, 0.f, 0.f};
        e = cudaGraphLaunch(ge, stream);  // warm-up
        for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
            cudaEventRecord(t0, stream);
            cudaGraphLaunch(ge, stream);
            cudaEventRecord(t1, stream);
            e = cudaEventSynchronize(t1);
            if (e == cudaSuccess) cudaEventElapsedTime(&times[rep], t0, t1);
        }
        cudaGraphExecDestroy(ge);
        if (e != cudaSuccess) break;
        std::sort(times, times + 3);
        const float per = times[1] / launches;
        if (getenv("MBW_LOG") && atoi(getenv("MBW_LOG")) >= 2)
            fprintf(stderr, "[mbw]   candidate %zu %s: %.3f us\n", ci, plan_to_string(op, p).c_str(), per * 1e3f);
        if (per < best_ms) {
            best_ms = per;
            best = p;
        }
    }
    if (stream) {
        cudaStreamSynchronize(stream);
        cudaStreamDestroy(stream);
    }
    if (t0) cudaEventDestroy(t0);
    if (t1) cudaEventDestroy(t1);
    if (wbuf) cudaFree(wbuf);
    if (xbuf) cudaFree(xbuf);
    if (ybuf) cudaFree(ybuf);
    if (nbuf) cudaFree(nbuf);
    if (rbuf) cudaFree(rbuf);
    if (e != cudaSuccess) {
        set_last_error(std::string("mbw_autotune: ") + cudaGetErrorString(e));
        return MBW_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        g_plans[key_of(op, M, N, K)] = best;
    }
    if (getenv("MBW_LOG")) {
        fprintf(stderr, "[mbw] autotune op=%d M=%lld N=%lld K=%lld -> %s (%.3f us)\n", op, (long long)M,
                (long long)N, (long long)K, plan_to_string(op, best).c_str(), best_ms * 1e3f);
    }
    return MBW_OK;
}
