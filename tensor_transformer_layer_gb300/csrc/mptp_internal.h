// Host-side helpers shared by the entry points: tensor-map encoding, device
// checks, the wait budget, and argument validation utilities.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "mptp.h"

namespace mptp {

// 2-D bf16 tensor map over a row-major [outer, inner] matrix with a row pitch of
// pitch_elems elements; box = box_inner x box_outer elements, 128-byte swizzle,
// zero fill out of bounds. Returns false if the driver rejects it.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                    uint32_t box_inner, uint32_t box_outer);

// Same with the 64-byte swizzle (boxes up to 32 bf16 wide).
bool make_tmap_bf16_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                         uint32_t box_inner, uint32_t box_outer);

// Tensor map for an epilogue output: 32 x 32 boxes, 64-byte swizzle (the layout
// the epilogue stages rows in before its TMA store).
// MN-major operand [outer rows, inner columns] as a 3-D map of 64-column blocks (SW128), box of
// 64 rows x `blocks` blocks; inner must be a multiple of 64.
bool make_tmap_bf16_mn3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
                         uint32_t blocks);
// MN-major GEMM operand [outer rows, inner columns] for CTA-pair tiles (two 64-wide blocks per
// CTA and stage): a 3-D map when inner is a multiple of 64 (returns majorness flag 2: one TMA box
// per stage), else 64-wide 2-D boxes (flag 1). 0: the map could not be encoded.
int make_tmap_mn_operand(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems);
bool make_tmap_bf16_out(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems);
// fp32 epilogue target [outer rows, inner columns] in 32 x 32 boxes (128-byte rows, 128-byte
// swizzle): the staging layout of the accumulating epilogue's TMA stores and reductions.
bool make_tmap_f32_out(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_elems);

// Unit order for a GEMM whose A operand (M side) has a_bytes and B operand (N side)
// b_bytes: walk the smaller operand's blocks fastest, so it stays resident in L2
// while concurrent CTAs share the slices of the larger one.
inline int n_fastest_order(double a_bytes, double b_bytes) { return b_bytes < a_bytes ? 1 : 0; }

// MP_OK if the current device is compute capability 10.3; fills the SM count.
mp_status check_device(int* num_sms);

// Bounded-wait budget for the kernels (ns): MPTP_WAIT_BUDGET_NS, default 2 s.
unsigned long long wait_budget_ns();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Cross-entropy partitioning: each of the t vocabulary shards (v_pad / t rows
// of E) is cut into equal chunks of whole BN-wide tiles for load balance; a unit of
// the logit kernel is one 256-token block times one chunk.
struct CePlan {
    int bn;              // 256 or 128
    int tiles_per_unit;  // tiles per chunk
    int chunk_cols;      // tiles_per_unit * bn
    int P;               // v_pad / chunk_cols partitions
};
// CTA pairs the plan balances the units over: the GB300's 152 SMs hold 76 pairs of the logit
// kernel. The plan depends on the sizes only (not on the device), so the workspace size and
// every entry point agree.
constexpr int CE_PLAN_PAIRS = 76;
// The plan for T tokens. Chunks of at least four tiles, or fewer tiles when that balances the
// units' last round at least 3 % better (T = 4096, v_pad = 51,200, t = 8: one-tile chunks,
// 43 rounds of one tile against 9 rounds of five). With workspace_limit > 0 and the preferred
// plan's triples larger than it: the cheapest plan that fits (else the fewest partitions).
bool ce_plan(int T, int v_pad, int t, size_t workspace_limit, CePlan* plan);
// Bytes of the triples of that plan (0 on invalid sizes).
size_t ce_plan_workspace(int T, int v_pad, int t, size_t workspace_limit);

// Two extra streams of the current device with fork/join events, for GEMMs that run
// side by side with the caller's stream; every launch on them is still ordered after
// the work the caller enqueued before (fork) and before the work it enqueues after
// (join). Created on first use outside a stream capture and kept for the process.
struct SideStreams {
    cudaStream_t s[2];
    cudaEvent_t fork;
    cudaEvent_t join[2];
};
// Hold side_stream_mutex() from side_streams() until the join has been enqueued.
std::mutex& side_stream_mutex();
// nullptr if they cannot be created now (no device, out of resources, or `origin` is
// being captured and they do not exist yet).
SideStreams* side_streams(cudaStream_t origin);

// Static split of `pairs` CTA pairs among n <= 3 GEMMs launched side by side. GEMM i has
// units[i] output tiles of cost[i] (K blocks plus the epilogue); on c pairs it takes
// ceil(units / c) rounds. Fills split[] and returns the makespan in cost units; a split
// never gives a GEMM more pairs than it has units.
long long split_pairs(int pairs, int n, const int* units, const int* cost, int* split);

// Makespan of the same GEMMs one after another, each on all `pairs`.
long long serial_makespan(int pairs, int n, const int* units, const int* cost);

}  // namespace mptp
