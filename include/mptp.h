/*
 * libmptp: the hot path of Megatron-LM intra-layer (tensor) model parallelism
 * on one GB300 (sm_103a) GPU.
 *
 * Two computations, both from "Megatron-LM: Training Multi-Billion Parameter
 * Language Models Using Model Parallelism" (paper-graph-ui summary), section 3.4
 * "Detailed, Sentence-Based Technical Breakdown", and from "Tensor and pipeline
 * parallelism, and choosing a layout" (ML Systems lesson 9), section 3,
 * Proposition (Megatron MLP split):
 *
 *   1. The partitioned MLP block Z = GeLU(X A) B with A split by columns and B by
 *      rows into t shards. The t shards live in one device's memory; the sum of
 *      the shard partials (the page's g all-reduce) and the sum of the shards'
 *      input gradients (the f all-reduce) are done inside the GEMM K-loop, which
 *      visits the shards in ascending order and accumulates in tensor memory.
 *   2. The vocab-parallel output GEMM fused with softmax cross-entropy: each
 *      vocabulary partition reduces its logits to a per-token (max, sum-exp,
 *      target-logit) triple; logits never reach global memory; a combine kernel
 *      turns the triples into the per-token loss.
 *
 * Conventions for every entry point
 *   - All matrices are bf16 (raw bits in mp_bf16), row-major and contiguous,
 *     except targets (int32), loss (fp32) and workspaces (opaque bytes).
 *   - All pointers are DEVICE pointers, 16-byte aligned. The caller allocates,
 *     owns and frees every buffer; the library never allocates and keeps no
 *     device memory between calls, with one exception: the static 4 MiB array
 *     of mp_vocab_ce_noalloc, which a device holds from that entry point's
 *     first call on it until the process exits.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work on it and return; nothing synchronises the host.
 *   - Argument and shape errors are reported synchronously, before any launch
 *     (nothing is enqueued). A failed launch returns MP_ERR_CUDA.
 *   - `d_status` (nullable, device memory, one uint32): conditions found on the
 *     device (MP_DEV_* bits) are OR-ed into it. The caller zeroes it before the
 *     call and reads it after synchronising the stream. With NULL they are not
 *     reported (outputs are still written as documented).
 *   - Every wait inside a kernel is bounded (default 2 s, environment variable
 *     MPTP_WAIT_BUDGET_NS overrides); when a bound runs out the kernel sets
 *     MP_DEV_TIMEOUT, lets its own copies and MMAs in flight finish, frees its
 *     tensor memory and returns. Outputs are then undefined.
 *   - Kernels are launched with programmatic stream serialization: a kernel may
 *     begin its set-up while the previous kernel in the stream finishes, and
 *     reads or writes global memory only after that kernel has completed, so
 *     stream order and CUDA-graph capture behave as for plain launches.
 *     MPTP_PDL=0 launches them plainly.
 *   - Outputs are overwritten, never accumulated into. T = 0 is a valid no-op.
 *   - Results are deterministic: no atomics in any reduction, fixed order.
 */
#ifndef MPTP_H
#define MPTP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MP_API __attribute__((visibility("default")))
#else
#define MP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mp_status {
    MP_OK = 0,
    MP_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad t */
    MP_ERR_UNSUPPORTED_SHAPE = 2, /* a size rule below is broken */
    MP_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
    MP_ERR_NO_DEVICE = 4,         /* current device is not compute capability 10.3 */
    MP_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
    MP_ERR_TIMEOUT = 6,           /* device bit MP_DEV_TIMEOUT was found (see mp_status_from_device) */
    MP_ERR_TARGET_RANGE = 7,      /* device bit MP_DEV_TARGET_RANGE was found */
    MP_ERR_WORKSPACE = 8          /* workspace too small */
} mp_status;

typedef uint16_t mp_bf16; /* raw bfloat16 bits */

/* Bits OR-ed into *d_status by the kernels. */
#define MP_DEV_TIMEOUT 0x1u
#define MP_DEV_TARGET_RANGE 0x2u

/*
 * Forward of the sharded MLP block.
 *   Column-parallel GEMM + GeLU (section 3.4 "Column-Parallel GEMM for the First
 *   MLP Layer"; Proposition steps 1-2): U = X A, Y = GeLU(U), exact erf form
 *   GeLU(u) = u (1 + erf(u / sqrt 2)) / 2, computed in fp32 from the fp32
 *   accumulator; all t column shards A_i = A[:, i f/t : (i+1) f/t] in one launch.
 *   Row-parallel GEMM + in-kernel g (section 3.4 "Row-Parallel GEMM for the
 *   Second MLP Layer"; Proposition step 3): Z = sum_i Y_i B_i, shards visited in
 *   ascending order, fp32 accumulation in tensor memory, one bf16 store.
 *
 *   X [T, h], A [h, f], B [f, h]            inputs
 *   Z [T, h]                                 output
 *   Y [T, f]                                 output (required): GeLU(U), bf16; read
 *                                            by the row-parallel GEMM and by mp_mlp_bwd
 *   U_save [T, f] or NULL                    output: U = X A rounded to bf16; needed
 *                                            by mp_mlp_bwd
 *   Size rules: T >= 0; h % 64 == 0; f % t == 0; (f / t) % 64 == 0; t >= 1.
 */
MP_API mp_status mp_mlp_fwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                     mp_bf16* Z, mp_bf16* Y, mp_bf16* U_save,
                     int T, int h, int f, int t,
                     uint32_t* d_status, void* stream);

/*
 * Backward of the sharded MLP block (Proposition steps 4-5), G = dZ:
 *   dU = (G B^T) * GeLU'(U), GeLU'(u) = Phi(u) + u phi(u), U read from U_save;
 *   dX = sum_i dU_i A_i^T  (the f operator's sum, fused into the K-loop, shards
 *                           in ascending order);
 *   dA = X^T dU  (all shards' dA_i side by side), dB = Y^T G.
 *
 *   X [T,h], A [h,f], B [f,h], U [T,f], Y [T,f], dZ [T,h]   inputs
 *   dX [T,h], dA [h,f], dB [f,h]                           outputs
 *   dU_ws [T,f]                                             workspace (caller-owned);
 *                                                           holds dU (bf16) on return
 *   Size rules as mp_mlp_fwd.
 *   Streams: everything is ordered on `stream`. When its estimated makespan is at
 *   least 6 % shorter, dX, dA and dB run side by side on disjoint CTA pairs, dX on
 *   `stream` and dA, dB on two internal side streams of the device that wait on an
 *   event recorded on `stream` and are joined back to it before the call returns
 *   (also inside a CUDA graph capture, once the side streams exist). The results are
 *   bitwise the same either way. MPTP_BWD_SCHEDULE=serial|overlap forces one of them.
 */
MP_API mp_status mp_mlp_bwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                     const mp_bf16* U, const mp_bf16* Y, const mp_bf16* dZ,
                     mp_bf16* dX, mp_bf16* dA, mp_bf16* dB, mp_bf16* dU_ws,
                     int T, int h, int f, int t,
                     uint32_t* d_status, void* stream);

/*
 * The same two computations for a range of shards [shard_begin, shard_begin +
 * shard_count) of the t shards: the work the GPUs holding those shards do before
 * the all-reduce ("Megatron-LM: Training Multi-Billion Parameter Language Models
 * Using Model Parallelism", section 3.4 "Row-Parallel GEMM for the Second MLP
 * Layer": each GPU's partial output, summed by g; "Megatron-LM, annotated",
 * section 3.1, "The second matrix: cut by rows, add once", which prints the two
 * partials of its one-token example). With c = [shard_begin f/t, (shard_begin +
 * shard_count) f/t):
 *   mp_mlp_fwd_shards:  Y[:, c] = GeLU(X A[:, c]) (and U_save[:, c]);
 *                       Z = sum over the range's shards i, ascending, of Y_i B_i
 *                       (the partial output; the full sum when the range is [0, t)).
 *   mp_mlp_bwd_shards:  dU_ws[:, c] = (dZ B[c, :]^T) * GeLU'(U[:, c]);
 *                       dX = sum over the range's shards i of dU_i A_i^T (the part
 *                       of dX those shards give before the f all-reduce);
 *                       dA[:, c] = X^T dU_ws[:, c];  dB[c, :] = Y[:, c]^T dZ.
 * Tensors are the full-size ones of mp_mlp_fwd / mp_mlp_bwd (shard i is a view);
 * only the range's columns of Y, U_save, dU_ws, dA and rows of dB are written, the
 * rest is left untouched. Each of those elements equals the full call's bit for
 * bit. Size rules as mp_mlp_fwd, and 0 <= shard_begin, 1 <= shard_count,
 * shard_begin + shard_count <= t (else MP_ERR_INVALID_ARG). mp_mlp_fwd and
 * mp_mlp_bwd are these calls with the range [0, t). A device that holds only its
 * own shards, contiguously, gets its partial from mp_mlp_fwd / mp_mlp_bwd with its
 * local f and t.
 */
MP_API mp_status mp_mlp_fwd_shards(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                            mp_bf16* Z, mp_bf16* Y, mp_bf16* U_save,
                            int T, int h, int f, int t, int shard_begin, int shard_count,
                            uint32_t* d_status, void* stream);
MP_API mp_status mp_mlp_bwd_shards(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                            const mp_bf16* U, const mp_bf16* Y, const mp_bf16* dZ,
                            mp_bf16* dX, mp_bf16* dA, mp_bf16* dB, mp_bf16* dU_ws,
                            int T, int h, int f, int t, int shard_begin, int shard_count,
                            uint32_t* d_status, void* stream);

/*
 * The MLP block with each direction in ONE kernel launch: the same computations
 * as mp_mlp_fwd_shards / mp_mlp_bwd_shards (same arguments, same outputs, equal
 * bit for bit), scheduled differently. In the forward, the row-parallel GEMM
 * (Z = sum_i Y_i B_i) starts on a block of 256 tokens as soon as the
 * column-parallel GEMM has written that block's rows of Y. In the backward, dX
 * (the f sum) starts on a block of tokens once its rows of dU exist, dA on a
 * 256-column tile of dU once that tile exists, and dB at once, on whichever SMs
 * are free. This is the overlap the method describes between the backward
 * all-reduce and the weight-gradient GEMMs ("Tensor and pipeline parallelism, and
 * choosing a layout", section 3, the remarks after the Proposition), inside one
 * grid, and it removes the part-empty last wave and the ramp of every GEMM but
 * the last.
 *
 *   workspace: mp_mlp_fused_workspace_bytes(T, h, f, t) bytes of device memory,
 *     16-byte aligned, ZERO-FILLED before its first use (e.g. cudaMemset once).
 *     It holds a few control words and one completion counter per 256-token row
 *     block and per 256-column tile of Y (dU). Every call returns it to zeros when
 *     its kernel ends, also after a timeout, so consecutive calls on one stream may
 *     share it (and a CUDA graph may replay a captured call). Smaller, NULL or
 *     misaligned: MP_ERR_WORKSPACE, nothing launched.
 *   Concurrency: a call's kernel takes every SM (one CTA pair per two SMs) and
 *     relies on all of its CTAs running at once, since a tile may wait for a tile of
 *     another CTA pair. Run these calls alone on the device; kernels enqueued before
 *     them on the same stream are fine. Beside another kernel on a different stream
 *     (or another of these calls), or where the process may use fewer SMs than the
 *     device has (an MPS limit on active threads), a CTA pair can wait for one that
 *     is not resident; the bounded wait then ends the call with MP_DEV_TIMEOUT
 *     instead of a hang. The separate-launch entry points have no such requirement.
 *   Size rules, shard range and outputs as mp_mlp_fwd_shards / mp_mlp_bwd_shards;
 *   dU_ws as mp_mlp_bwd. T = 0: nothing to compute (the backward zeroes its dA and
 *   dB range, as mp_mlp_bwd_shards does) and the workspace is not touched.
 *   Large layers run as mp_mlp_fwd_shards / mp_mlp_bwd_shards do, as separate
 *   launches with the same outputs, and leave the workspace untouched: a direction
 *   with more than 4096 output tiles of 256 x 256 (at h = 3072: the backward beyond
 *   about 12.5k tokens, the forward beyond about 17k), and any layer with T > 8192
 *   and h < 2304, where one launch measured 1-7 % slower than the separate ones.
 */
MP_API size_t mp_mlp_fused_workspace_bytes(int T, int h, int f, int t);
MP_API mp_status mp_mlp_fwd_fused(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                           mp_bf16* Z, mp_bf16* Y, mp_bf16* U_save,
                           int T, int h, int f, int t, int shard_begin, int shard_count,
                           void* workspace, size_t workspace_bytes,
                           uint32_t* d_status, void* stream);
MP_API mp_status mp_mlp_bwd_fused(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B,
                           const mp_bf16* U, const mp_bf16* Y, const mp_bf16* dZ,
                           mp_bf16* dX, mp_bf16* dA, mp_bf16* dB, mp_bf16* dU_ws,
                           int T, int h, int f, int t, int shard_begin, int shard_count,
                           void* workspace, size_t workspace_bytes,
                           uint32_t* d_status, void* stream);

/*
 * Bytes of workspace mp_vocab_ce needs for its fastest partition: fp32 triples
 * [P][3][T], P = the number of vocabulary partitions (the t shards, each cut into
 * equal chunks of whole tiles; the chunk size balances the logit kernel's units
 * over the GPU for this T, e.g. P = 40 at T = 8192 and 200 at T = 4096 for
 * v_pad = 51,200, t = 8). A smaller workspace also works down to one partition
 * per shard (12 t T bytes): the entry points then take the fastest partition
 * that fits it (mp_vocab_ce_partials and mp_vocab_ce_combine must be given the
 * same workspace size). Returns 0 on invalid sizes.
 */
MP_API size_t mp_vocab_ce_workspace_bytes(int T, int v_pad, int t);

/*
 * Vocab-parallel output GEMM fused with softmax cross-entropy
 * (section 3.4 "Output Embedding Parallelism and the Fused Cross-Entropy
 * Optimization", steps 1-6).
 *   Logits z[r, c] = X[r] . E[c] for c in [0, v_valid); padding rows
 *   c >= v_valid ("Vocabulary padding for efficiency") are excluded.
 *   loss[r] = M + log(S) - z[r, target[r]], M = max_c z, S = sum_c exp(z - M).
 *
 *   X [T, h] bf16, E [v_pad, h] bf16 (the vocabulary split into t row blocks of
 *   v_pad / t), target [T] int32 in [0, v_valid), loss [T] fp32 output,
 *   workspace: mp_vocab_ce_workspace_bytes(T, v_pad, t) bytes (fp32 triples), or
 *   fewer down to 12 t T bytes (a coarser partition; MP_ERR_WORKSPACE below that).
 *   Size rules: h % 64 == 0; t >= 1; v_pad % (128 t) == 0; 1 <= v_valid <= v_pad.
 *   A target outside [0, v_valid) sets MP_DEV_TARGET_RANGE and gives NaN loss for
 *   that token; nothing is read out of bounds.
 */
MP_API mp_status mp_vocab_ce(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                      float* loss, void* workspace, size_t workspace_bytes,
                      int T, int h, int v_pad, int v_valid, int t,
                      uint32_t* d_status, void* stream);

/* First half of mp_vocab_ce: the logit GEMM whose epilogue writes the per-token,
 * per-partition (max, sum-exp, target-logit) triples into workspace (steps 1-4). */
MP_API mp_status mp_vocab_ce_partials(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                               void* workspace, size_t workspace_bytes,
                               int T, int h, int v_pad, int v_valid, int t,
                               uint32_t* d_status, void* stream);

/* Second half of mp_vocab_ce: combine the triples into loss (steps 5-6):
 * M = max_p m_p, S = sum_p s_p exp(m_p - M), loss = M + log S - z_target. */
MP_API mp_status mp_vocab_ce_combine(const void* workspace, size_t workspace_bytes,
                              const int32_t* target, float* loss,
                              int T, int v_pad, int v_valid, int t,
                              uint32_t* d_status, void* stream);

/* mp_vocab_ce that also writes the per-token log-sum-exp over the valid vocabulary,
 * lse[r] = M + log S (fp32 [T], device memory, required when T > 0), the quantity the
 * backward needs (mp_vocab_ce_bwd_lse). lse is NaN for a token whose target is outside
 * [0, v_valid) (that token contributes no gradient). loss is bit for bit mp_vocab_ce's. */
MP_API mp_status mp_vocab_ce_lse(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                          float* loss, float* lse, void* workspace, size_t workspace_bytes,
                          int T, int h, int v_pad, int v_valid, int t,
                          uint32_t* d_status, void* stream);

/*
 * Backward of the vocab-parallel cross-entropy. The pages describe the fused
 * forward only; this is the plain derivative of softmax cross-entropy, computed
 * in the forward's vocabulary partition so that logit gradients exist for one
 * shard (v_pad / t columns) at a time:
 *   dZ[r, c] = dloss[r] * (softmax(z[r])_c - [c == target[r]]) for c < v_valid,
 *   0 for padding columns;  dX = dZ E;  dE = dZ^T X  (padding rows of dE are 0).
 * The per-token log-sum-exp is taken from the forward's loss:
 *   lse[r] = loss[r] + X[r] . E[target[r]].
 *
 *   X [T, h] bf16, E [v_pad, h] bf16, target [T] int32, loss [T] fp32 (the output of
 *   mp_vocab_ce on the same X, E, target), dloss [T] fp32 (upstream gradient, e.g.
 *   1/T for a mean) -> dX [T, h] bf16, dE [v_pad, h] bf16 (overwritten).
 *   workspace >= mp_vocab_ce_bwd_workspace_bytes(T, h, v_pad, t) bytes: the
 *   log-sum-exp [T], a few hundred bytes of counters (the call zeroes them), an fp32
 *   dX accumulator [T, h] and one shard of dZ [T, v_pad/t]; no initial value needed.
 *   The shards are processed one after another, each shard's three GEMMs in ONE
 *   kernel launch (dX and dE tiles start as soon as the dZ rows or columns they read
 *   exist). That launch takes every SM and relies on all of its CTAs running at once,
 *   so the same concurrency rule as mp_mlp_fwd_fused applies: run it alone on the
 *   device (beside other kernels it ends with MP_DEV_TIMEOUT rather than hang).
 *   MPTP_CE_BWD_CHAIN=0 in the environment runs each shard as three separate
 *   launches instead, with no such rule (so does a shard with more than 4096 output
 *   tiles, about T > 32k tokens at v_pad / t = 6400); the gradients are the same bit
 *   for bit.
 *   workspace >= mp_vocab_ce_bwd_workspace_bytes_one_pass(T, h, v_pad, t) bytes
 *   (the log-sum-exp and every shard's dZ, [T, v_pad] bf16: 839 MB at T = 8192,
 *   v_pad = 51,200): dZ of all shards is formed in one launch, then dE and dX in
 *   one GEMM each, dX accumulating the shards inside its K-loop (no fp32 round
 *   trips); faster, same results within rounding.
 *   Size rules as mp_vocab_ce. A target outside [0, v_valid) sets
 *   MP_DEV_TARGET_RANGE and contributes no gradient. dX sums the shards in
 *   ascending order (deterministic for a given workspace size).
 */
MP_API size_t mp_vocab_ce_bwd_workspace_bytes(int T, int h, int v_pad, int t);
MP_API size_t mp_vocab_ce_bwd_workspace_bytes_one_pass(int T, int h, int v_pad, int t);
MP_API mp_status mp_vocab_ce_bwd(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                          const float* loss, const float* dloss,
                          mp_bf16* dX, mp_bf16* dE, void* workspace, size_t workspace_bytes,
                          int T, int h, int v_pad, int v_valid, int t,
                          uint32_t* d_status, void* stream);

/* mp_vocab_ce_bwd from the forward's exported log-sum-exp (mp_vocab_ce_lse) instead of its
 * loss: no recompute of the target logits (one launch fewer). Same workspace sizes, outputs
 * and rules; a NaN lse marks a token with an invalid target, which gets no gradient (the
 * forward set MP_DEV_TARGET_RANGE for it). */
MP_API mp_status mp_vocab_ce_bwd_lse(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                              const float* lse, const float* dloss,
                              mp_bf16* dX, mp_bf16* dE, void* workspace, size_t workspace_bytes,
                              int T, int h, int v_pad, int v_valid, int t,
                              uint32_t* d_status, void* stream);

/*
 * Vocab-parallel input embedding ("Megatron-LM: Training Multi-Billion Parameter
 * Language Models Using Model Parallelism", section 3.4 "Input Embedding
 * Parallelism"): E [v_pad, h] split along the vocabulary into t shards of v_pad/t
 * rows; each shard looks up the ids in its range (zeros elsewhere) and the shards'
 * results are summed (the g all-reduce). One shard owns each valid id, so
 *   out[r] = E[ids[r]] exactly (bit for bit) for ids in [0, v_valid);
 *   out[r] = 0 and MP_DEV_TARGET_RANGE set for any other id (no shard owns it).
 *   ids [T] int32, E [v_pad, h] bf16, out [T, h] bf16 (overwritten).
 *   Size rules: h % 64 == 0; t >= 1; v_pad % (128 t) == 0; 1 <= v_valid <= v_pad.
 */
MP_API mp_status mp_vocab_embed(const int32_t* ids, const mp_bf16* E, mp_bf16* out,
                         int T, int h, int v_pad, int v_valid, int t,
                         uint32_t* d_status, void* stream);

/*
 * Forward of the head-parallel self-attention block ("Megatron-LM: Training
 * Multi-Billion Parameter Language Models Using Model Parallelism", section 3.4
 * "Attention Head Parallelism in the Self-Attention Block"; "Megatron-LM,
 * annotated", section 3.2): heads are split across t shards by the columns of the
 * Q, K, V projections; each head runs causal softmax attention (GPT-2 decoder);
 * the output projection is split by rows and the shards' partials are summed (g).
 *   QKV = X Wqkv;  O[:, head j] = softmax(Q_j K_j^T / sqrt(d) + causal) V_j;
 *   out = sum_i O_i Wo_i (shards in ascending order inside the GEMM K-loop).
 *   X [b s, h] (b sequences of s tokens), Wqkv [h, 3h] = [Wq | Wk | Wv] with head j at
 *   columns [j d, (j+1) d) of each, Wo [h, h]; outputs QKV [b s, 3h], O [b s, h] (both
 *   kept for a backward pass) and out [b s, h], bf16, overwritten.
 *   Size rules: d = h / heads in {64, 96}; heads % t == 0; h % 64 == 0; s % 128 == 0.
 */
MP_API mp_status mp_attn_fwd(const mp_bf16* X, const mp_bf16* Wqkv, const mp_bf16* Wo,
                      mp_bf16* out, mp_bf16* QKV, mp_bf16* O,
                      int b, int s, int h, int heads, int t,
                      uint32_t* d_status, void* stream);

/*
 * mp_vocab_ce for callers that cannot allocate device memory. The paper has no
 * counterpart to this entry point; it exists for callers whose device memory is
 * owned by another pool (a serving runtime that reserves HBM at start-up and
 * forbids later cudaMalloc/cudaFree, which can synchronise the device; a host
 * framework that must account for every byte), so they cannot pass a workspace.
 *
 * Same inputs, outputs and size rules as mp_vocab_ce, without the workspace: the
 * triples live in a static device array of MP_CE_NOALLOC_MAX_FLOATS floats
 * (4 MiB), held by every GPU the entry point has run on, until exit.
 *   - The vocabulary partition is the fastest one whose triples fit in 4 MiB
 *     (the same as mp_vocab_ce's when mp_vocab_ce_workspace_bytes(T, v_pad, t)
 *     <= 4 MiB, e.g. T <= 8738 at v_pad = 51,200, t = 8 apart from small T).
 *     Problems that fit in no partition (one per shard: 12 t T bytes > 4 MiB,
 *     e.g. T > 43,690 at t = 8) return MP_ERR_WORKSPACE before any launch.
 *   - Nothing is allocated by the call: no cudaMalloc, cudaFree or allocating
 *     library call. CUDA itself places the array on a device when it loads the
 *     code that holds it, which with lazy module loading (the default) is this
 *     entry point's first call on that device, T = 0 included. Make one call
 *     (T = 0 suffices) with the device current before a memory pool reserves
 *     the rest of HBM and before any stream capture, or run the process with
 *     CUDA_MODULE_LOADING=EAGER.
 *   - Every call looks up the array's device address with the current device
 *     (a host-side query), so it stays valid after cudaDeviceReset.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (nothing in it needs to start at zero). Calls whose work overlaps
 *     on the GPU (other streams, other host threads) race on it: serialise them.
 *   - If the logit kernel gives up on a bounded wait it writes no triples, and
 *     the losses may then be computed from the previous call's triples: they can
 *     look valid. Pass d_status and check it for MP_DEV_TIMEOUT.
 */
#define MP_CE_NOALLOC_MAX_FLOATS (1024 * 1024)
MP_API mp_status mp_vocab_ce_noalloc(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                              float* loss, int T, int h, int v_pad, int v_valid, int t,
                              uint32_t* d_status, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
MP_API const char* mp_status_string(mp_status s);

/* Map device status bits to the status code a caller should report
 * (MP_OK when bits == 0; timeout takes precedence). */
MP_API mp_status mp_status_from_device(uint32_t bits);

/* Library version, major * 10000 + minor * 100 + patch. */
MP_API int mp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MPTP_H */
