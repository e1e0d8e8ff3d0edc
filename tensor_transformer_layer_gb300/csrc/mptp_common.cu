// Status strings, tensor-map encoding through the driver entry point, the
// device check and the wait budget.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "mptp_internal.h"

namespace mptp {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

static bool make_tmap_bf16_sw(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                    uint32_t box_inner, uint32_t box_outer) {
    return make_tmap_bf16_sw(map, base, inner, outer, pitch_elems, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                         uint32_t box_inner, uint32_t box_outer) {
    return make_tmap_bf16_sw(map, base, inner, outer, pitch_elems, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tmap_bf16_mn3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                         uint32_t blocks) {
    auto fn = encode_fn();
    if (fn == nullptr || inner % 64 != 0) return false;
    // (column within a 64-wide block, row, block): a box of 64 rows x `blocks` blocks lands as
    // `blocks` consecutive 64-row x 128-byte slabs, the layout of as many 2-D boxes.
    cuuint64_t dims[3] = {64, outer, inner / 64};
    cuuint64_t strides[2] = {pitch_elems * 2, 128};
    cuuint32_t box[3] = {64, 64, blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int make_tmap_mn_operand(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems) {
    if (inner % 64 == 0) return make_tmap_bf16_mn3d(map, base, inner, outer, pitch_elems, 2) ? 2 : 0;
    return make_tmap_bf16(map, base, inner, outer, pitch_elems, 64, 64) ? 1 : 0;
}

bool make_tmap_bf16_out(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems) {
    return make_tmap_bf16_sw(map, base, inner, outer, pitch_elems, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tmap_f32_out(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_elems * 4};
    cuuint32_t box[2] = {32, 32};  // 32 rows of 128 bytes
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

mp_status check_device(int* num_sms) {
    constexpr int MAXDEV = 64;
    static std::atomic<int> cached[MAXDEV];  // 0 unknown, -1 bad, >0 SM count
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MP_ERR_NO_DEVICE;
    }
    if (dev >= 0 && dev < MAXDEV) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *num_sms = c;
            return MP_OK;
        }
        if (c < 0) return MP_ERR_NO_DEVICE;
    }
    int maj = 0, min = 0, sms = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MP_ERR_NO_DEVICE;
    }
    const bool ok = (maj == 10 && min == 3 && sms > 0);
    if (dev >= 0 && dev < MAXDEV) cached[dev].store(ok ? sms : -1, std::memory_order_relaxed);
    if (!ok) return MP_ERR_NO_DEVICE;
    *num_sms = sms;
    return MP_OK;
}

unsigned long long wait_budget_ns() {
    const char* s = std::getenv("MPTP_WAIT_BUDGET_NS");
    if (s != nullptr && *s) {
        char* end = nullptr;
        const unsigned long long v = std::strtoull(s, &end, 10);
        if (end != s) return v;
    }
    return 2000000000ull;
}

static void ce_plan_with(int v_pad, int t, int tpu, CePlan* plan) {
    const int vs = v_pad / t;
    plan->bn = (vs % 256 == 0) ? 256 : 128;
    plan->tiles_per_unit = tpu;
    plan->chunk_cols = tpu * plan->bn;
    plan->P = v_pad / plan->chunk_cols;
}

static size_t ce_plan_bytes(int T, const CePlan& p) { return size_t(p.P) * 3 * size_t(T) * sizeof(float); }

bool ce_plan(int T, int v_pad, int t, size_t workspace_limit, CePlan* plan) {
    if (T < 0 || t < 1 || v_pad < 128 * t || v_pad % (128 * t) != 0) return false;
    const int vs = v_pad / t;
    const int bn = (vs % 256 == 0) ? 256 : 128;
    const int nb = vs / bn;  // tiles per shard
    // The default chunk: the smallest divisor of nb that is at least 4 tiles (or the whole shard).
    int base = nb;
    for (int d = 4; d <= nb; ++d)
        if (nb % d == 0) {
            base = d;
            break;
        }
    // Estimated time in tile-times on CE_PLAN_PAIRS pairs: rounds of units x tiles per unit.
    const long long mblocks = (static_cast<long long>(T) + 255) / 256;
    auto cost = [&](int tpu) {
        const long long units = mblocks * (v_pad / (tpu * bn));
        return (units + CE_PLAN_PAIRS - 1) / CE_PLAN_PAIRS * tpu;
    };
    // Preferred: the default, or a finer divisor that is at least 3 % cheaper (more partitions
    // balance the last round of units); fewer tiles per unit only when it pays.
    int pick = base;
    for (int d = 1; d < base; ++d)
        if (nb % d == 0 && cost(d) * 100 <= cost(base) * 97 && cost(d) < cost(pick)) pick = d;
    ce_plan_with(v_pad, t, pick, plan);
    if (workspace_limit == 0 || ce_plan_bytes(T, *plan) <= workspace_limit) return true;
    // A smaller workspace: the cheapest plan that fits, else the one with the fewest partitions.
    int fit = 0;
    for (int d = 1; d <= nb; ++d) {
        if (nb % d != 0) continue;
        CePlan c;
        ce_plan_with(v_pad, t, d, &c);
        if (ce_plan_bytes(T, c) <= workspace_limit && (fit == 0 || cost(d) < cost(fit) || (cost(d) == cost(fit) && d > fit)))
            fit = d;
    }
    ce_plan_with(v_pad, t, fit > 0 ? fit : nb, plan);
    return true;
}

size_t ce_plan_workspace(int T, int v_pad, int t, size_t workspace_limit) {
    CePlan plan;
    if (!ce_plan(T, v_pad, t, workspace_limit, &plan)) return 0;
    return ce_plan_bytes(T, plan);
}

namespace {
struct SideEntry {
    bool tried;
    bool ok;
    SideStreams ss;
};
std::mutex g_side_mu;
SideEntry g_side[64];
}  // namespace

std::mutex& side_stream_mutex() { return g_side_mu; }

SideStreams* side_streams(cudaStream_t origin) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    SideEntry& e = g_side[dev];
    if (!e.tried) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(origin, &cs) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        if (cs != cudaStreamCaptureStatusNone) return nullptr;
        e.tried = true;
        bool ok = true;
        for (int i = 0; i < 2; ++i)
            ok = ok && cudaStreamCreateWithFlags(&e.ss.s[i], cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&e.ss.fork, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < 2; ++i)
            ok = ok && cudaEventCreateWithFlags(&e.ss.join[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) cudaGetLastError();
        e.ok = ok;
    }
    return e.ok ? &e.ss : nullptr;
}

static long long rounds_cost(int units, int c, int cost) {
    return static_cast<long long>((units + c - 1) / c) * cost;
}

long long split_pairs(int pairs, int n, const int* units, const int* cost, int* split) {
    long long best = -1;
    int c[3] = {1, 1, 1};
    const int c0_max = pairs - (n - 1);
    for (c[0] = 1; c[0] <= c0_max; ++c[0]) {
        const int c1_max = n > 1 ? pairs - c[0] - (n - 2) : 1;
        for (c[1] = 1; c[1] <= c1_max; ++c[1]) {
            if (n > 2) c[2] = pairs - c[0] - c[1];
            long long span = 0;
            int use[3];
            for (int i = 0; i < n; ++i) {
                use[i] = c[i] < units[i] ? c[i] : units[i];
                const long long r = rounds_cost(units[i], use[i], cost[i]);
                span = r > span ? r : span;
            }
            if (best < 0 || span < best) {
                best = span;
                for (int i = 0; i < n; ++i) split[i] = use[i];
            }
            if (n == 1) break;
        }
    }
    return best;
}

long long serial_makespan(int pairs, int n, const int* units, const int* cost) {
    long long t = 0;
    for (int i = 0; i < n; ++i) t += rounds_cost(units[i], units[i] < pairs ? units[i] : pairs, cost[i]);
    return t;
}

}  // namespace mptp

extern "C" const char* mp_status_string(mp_status s) {
    switch (s) {
        case MP_OK: return "MP_OK";
        case MP_ERR_INVALID_ARG: return "MP_ERR_INVALID_ARG: null pointer, negative size or bad shard count";
        case MP_ERR_UNSUPPORTED_SHAPE: return "MP_ERR_UNSUPPORTED_SHAPE: a size rule of the entry point is broken";
        case MP_ERR_MISALIGNED: return "MP_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case MP_ERR_NO_DEVICE: return "MP_ERR_NO_DEVICE: current device is not compute capability 10.3 (sm_103a)";
        case MP_ERR_CUDA: return "MP_ERR_CUDA: a CUDA call failed";
        case MP_ERR_TIMEOUT: return "MP_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
        case MP_ERR_TARGET_RANGE: return "MP_ERR_TARGET_RANGE: a target id is outside [0, v_valid)";
        case MP_ERR_WORKSPACE: return "MP_ERR_WORKSPACE: workspace smaller than required";
    }
    return "MP_ERR_UNKNOWN";
}

extern "C" mp_status mp_status_from_device(uint32_t bits) {
    if (bits & MP_DEV_TIMEOUT) return MP_ERR_TIMEOUT;
    if (bits & MP_DEV_TARGET_RANGE) return MP_ERR_TARGET_RANGE;
    return MP_OK;
}

extern "C" int mp_version(void) { return 100; }
