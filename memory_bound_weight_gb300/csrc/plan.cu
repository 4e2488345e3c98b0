// plan.cu -- launch-time plan selection for the streaming GEMV kernels.
//
// A plan is (kernel instantiation, split-K cluster size). The default plan is a
// heuristic; mbw_autotune() replaces it by measurement, in the manner of
// tinyinfer's load-time autotuner ("R rows per warp" section: time R = 1, 2, 4
// on every distinct matrix shape at model load and keep the fastest, in a few
// milliseconds). Here the candidates are every kernel instantiation of the
// format x split factor {1, 2, 4, 8}; each is timed as a CUDA graph of
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

static int fmt_of_op(int op) {
    switch (op) {
        case MBW_OP_GEMV_INT4_G64: return FMT_G64;
        case MBW_OP_GEMV_INT4_AWQ_G128: return FMT_AWQ;
        default: return FMT_BF16;
    }
}

static int chunks_of(int fmt, int64_t K) { return (int)(fmt == FMT_BF16 ? K / 8 : K / 32); }

static size_t smem_needed(int fmt, const SimtConfig& c, int64_t K, int split) {
    GemvArgs a{};
    a.chunks = chunks_of(fmt, K);
    a.split_chunks = (a.chunks + split - 1) / split;
    return simt_smem_bytes(fmt, c, a, split);
}

static const size_t kSmemLimit = 200 * 1024;

// Batch width the call should use: the smallest kernel batch >= min(M, 8).
static int want_mb(int64_t M) { return M <= 2 ? (int)M : M <= 4 ? 4 : 8; }

static bool plan_valid(int fmt, const Plan& p, int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (p.cfg < 0 || p.cfg >= simt_num_configs(fmt)) return false;
    const SimtConfig c = simt_config(fmt, p.cfg);
    if (c.mb != want_mb(M)) return false;
    if (p.split < 1 || p.split > 8) return false;
    if (smem_needed(fmt, c, K, p.split) > kSmemLimit) return false;
    const int chunks = chunks_of(fmt, K);
    if (p.split > 1 && (chunks + p.split - 1) / p.split < 16) return false;
    return true;
}

Plan plan_default(int op, int64_t M, int64_t N, int64_t K) {
    const int fmt = fmt_of_op(op);
    const int mb = want_mb(M);
    // preferred instantiation per format and batch width
    int cfg = -1;
    const int n = simt_num_configs(fmt);
    const int pref_r = (fmt == FMT_BF16) ? 1 : 2;
    for (int i = 0; i < n && cfg < 0; ++i) {
        const SimtConfig c = simt_config(fmt, i);
        if (c.mb == mb && c.warps == 4 && (mb > 1 || c.r == pref_r)) cfg = i;
    }
    for (int i = 0; i < n && cfg < 0; ++i)
        if (simt_config(fmt, i).mb == mb) cfg = i;
    const SimtConfig c = simt_config(fmt, cfg);
    const int sms = device_sm_count();
    const int64_t rowblocks = (N + c.warps * c.r - 1) / (c.warps * c.r);
    const int chunks = chunks_of(fmt, K);
    int split = 1;
    while (split < 8 && (rowblocks * split < 2 * sms || smem_needed(fmt, c, K, split) > kSmemLimit) &&
           chunks / (2 * split) >= 32)
        split *= 2;
    while (split < 8 && smem_needed(fmt, c, K, split) > kSmemLimit) split *= 2;
    Plan p;
    p.kind = PLAN_SIMT;
    p.cfg = cfg;
    p.split = split;
    return p;
}

static int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

Plan plan_lookup(int op, int64_t M, int64_t N, int64_t K, cudaStream_t s) {
    (void)s;
    const auto key = std::make_tuple(current_device(), op, std::min<int64_t>(M, 8), N, K);
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
    const int fmt = fmt_of_op(op);
    const SimtConfig c = simt_config(fmt, p.cfg);
    char buf[160];
    snprintf(buf, sizeof(buf), "simt fmt=%s warps=%d rows_per_warp=%d chunks_in_flight=%d batch=%d split_k=%d",
             fmt == FMT_BF16 ? "bf16" : fmt == FMT_G64 ? "int4_g64" : "int4_awq_g128", c.warps, c.r, c.u, c.mb,
             p.split);
    return buf;
}

static size_t weight_bytes(int fmt, int64_t N, int64_t K) {
    if (fmt == FMT_BF16) return (size_t)N * K * 2;
    if (fmt == FMT_G64) return (size_t)N * K / 2 + (size_t)N * (K / 64) * 2;
    const int64_t G = K / 128;
    return (size_t)N * K / 2 + (size_t)N * G * 2 + (size_t)N * ((G + 1) / 2);
}

}  // namespace mbw

using namespace mbw;

extern "C" mbw_status mbw_plan_describe(int op, int64_t M, int64_t N, int64_t K, char* buf, size_t len) {
    if (!buf || len == 0) return MBW_ERR_INVALID_ARG;
    if (op < MBW_OP_GEMV_BF16 || op > MBW_OP_GEMM_SKINNY_BF16 || M < 1 || N < 1 || K < 1) {
        set_last_error("mbw_plan_describe: bad op or shape");
        return MBW_ERR_INVALID_ARG;
    }
    const Plan p = plan_lookup(op, M, N, K, nullptr);
    const std::string s = plan_to_string(op, p);
    snprintf(buf, len, "%s", s.c_str());
    return MBW_OK;
}

static std::vector<Plan> candidates(int op, int64_t M, int64_t N, int64_t K) {
    std::vector<Plan> out;
    const int fmt = fmt_of_op(op);
    const int64_t Mb = std::min<int64_t>(M, 8);
    const int splits[4] = {1, 2, 4, 8};
    for (int cfg = 0; cfg < simt_num_configs(fmt); ++cfg)
        for (int si = 0; si < 4; ++si) {
            Plan p;
            p.kind = PLAN_SIMT;
            p.cfg = cfg;
            p.split = splits[si];
            if (plan_valid(fmt, p, Mb, N, K)) out.push_back(p);
        }
    return out;
}

static bool shape_ok(int op, int64_t M, int64_t N, int64_t K) {
    if (op < MBW_OP_GEMV_BF16 || op > MBW_OP_GEMM_SKINNY_BF16) return false;
    if (M < 1 || N < 1 || K < 1 || N > 0x7FFFFFFF || K > 0x7FFFFFFF || M > 0x7FFFFFFF) return false;
    const int fmt = fmt_of_op(op);
    const int64_t kunit = fmt == FMT_BF16 ? 8 : fmt == FMT_G64 ? 64 : 128;
    return K % kunit == 0;
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
        if (c[i].kind == cur.kind && c[i].cfg == cur.cfg && c[i].split == cur.split) return (int)i;
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
    const auto key = std::make_tuple(current_device(), op, std::min<int64_t>(M, 8), N, K);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[key] = c[index];
    return MBW_OK;
}

extern "C" mbw_status mbw_autotune(int op, int64_t M, int64_t N, int64_t K, mbw_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!shape_ok(op, M, N, K)) {
        set_last_error("mbw_autotune: bad op or shape");
        return MBW_ERR_INVALID_ARG;
    }
    const int fmt = fmt_of_op(op);
    cudaStreamCaptureStatus cs;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone) {
        set_last_error("mbw_autotune: stream is capturing");
        return MBW_ERR_INVALID_ARG;
    }
    // Timing graphs are captured on a private stream (the caller's may be the
    // legacy default stream, which cannot be captured); the caller's stream
    // is drained first so that tuning does not overlap its work.
    cudaError_t se = cudaStreamSynchronize(stream);
    if (se != cudaSuccess) {
        set_last_error(std::string("mbw_autotune: ") + cudaGetErrorString(se));
        return MBW_ERR_CUDA;
    }
    cudaStream_t user_stream = stream;
    se = cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
    if (se != cudaSuccess) {
        set_last_error(std::string("mbw_autotune: ") + cudaGetErrorString(se));
        return MBW_ERR_CUDA;
    }
    const int64_t Mb = std::min<int64_t>(M, 8);
    const size_t wb = weight_bytes(fmt, N, K);
    const size_t wstride = (wb + 255) / 256 * 256;
    const size_t target = (size_t)384 << 20;  // well above the 126 MB L2
    int copies = (int)std::max<size_t>(2, (target + wb - 1) / wb);
    copies = std::min(copies, 96);

    uint8_t* wbuf = nullptr;
    uint16_t* xbuf = nullptr;
    void* ybuf = nullptr;
    cudaError_t e = cudaMalloc(&wbuf, wstride * copies);
    if (e == cudaSuccess) e = cudaMalloc(&xbuf, (size_t)Mb * K * 2);
    if (e == cudaSuccess) e = cudaMalloc(&ybuf, (size_t)Mb * N * 4);
    if (e == cudaSuccess) e = cudaMemsetAsync(wbuf, 0x37, wstride * copies, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(xbuf, 0x37, (size_t)Mb * K * 2, stream);
    cudaEvent_t t0 = nullptr, t1 = nullptr;
    if (e == cudaSuccess) e = cudaEventCreate(&t0);
    if (e == cudaSuccess) e = cudaEventCreate(&t1);

    Plan best = plan_default(op, M, N, K);
    float best_ms = 1e30f;
    const std::vector<Plan> cands = candidates(op, M, N, K);
    for (size_t ci = 0; ci < cands.size() && e == cudaSuccess; ++ci) {
        {
            const Plan p = cands[ci];
            GemvArgs a{};
            a.N = (int)N;
            a.K = (int)K;
            a.M = (int)Mb;
            a.x = xbuf;
            a.y = ybuf;
            a.chunks = chunks_of(fmt, K);
            a.split_chunks = (a.chunks + p.split - 1) / p.split;
            a.groups = (int)(fmt == FMT_G64 ? K / 64 : fmt == FMT_AWQ ? K / 128 : 0);
            a.zstride = (a.groups + 1) / 2;
            a.out_f32 = 0;
            const size_t codes = fmt == FMT_BF16 ? (size_t)N * K * 2 : (size_t)N * K / 2;
            cudaGraph_t g = nullptr;
            cudaGraphExec_t ge = nullptr;
            e = cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal);
            if (e != cudaSuccess) break;
            cudaError_t le = cudaSuccess;
            for (int i = 0; i < copies && le == cudaSuccess; ++i) {
                a.W = wbuf + (size_t)i * wstride;
                a.scales = (const uint16_t*)(a.W + codes);
                a.zeros = (const uint8_t*)(a.W + codes + (size_t)N * a.groups * 2);
                le = launch_gemv_simt(fmt, p, a, stream);
            }
            e = cudaStreamEndCapture(stream, &g);
            if (le != cudaSuccess || e != cudaSuccess) {
                // an invalid candidate (e.g. cluster shape not schedulable): skip it
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
            float times[3];
            cudaGraphLaunch(ge, stream);  // warm-up
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
            const float per = times[1] / copies;
            if (per < best_ms) {
                best_ms = per;
                best = p;
            }
        }
    }
    cudaStreamSynchronize(stream);
    cudaStreamDestroy(stream);
    (void)user_stream;
    if (t0) cudaEventDestroy(t0);
    if (t1) cudaEventDestroy(t1);
    if (wbuf) cudaFree(wbuf);
    if (xbuf) cudaFree(xbuf);
    if (ybuf) cudaFree(ybuf);
    if (e != cudaSuccess) {
        set_last_error(std::string("mbw_autotune: ") + cudaGetErrorString(e));
        return MBW_ERR_CUDA;
    }
    const auto key = std::make_tuple(current_device(), op, Mb, N, K);
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[key] = best;
    if (getenv("MBW_LOG")) {
        fprintf(stderr, "[mbw] autotune op=%d M=%lld N=%lld K=%lld -> %s (%.3f us)\n", op, (long long)M,
                (long long)N, (long long)K, plan_to_string(op, best).c_str(), best_ms * 1e3f);
    }
    return MBW_OK;
}
