/*
 * csbp.h -- C ABI of libcsbp: two-copy block-diffusion attention, forward and
 * backward, on one sm_103a GPU, with the per-rank math of context-sharded
 * block parallelism (CSBP) run as virtual clean shards.
 *
 * Method (sources, cited by page title and section):
 *  - "CSBP 完全拆解：块并行如何让长上下文扩散语言模型少传无效 KV" (blog),
 *    section "传统上下文并行为什么会传错东西": the input is a clean copy and a
 *    corrupted copy of a length-L sequence cut into B = L/M blocks; a
 *    corrupted query of block b reads exactly [K_b; K^clean_<b] and
 *    [V_b; V^clean_<b]; O = softmax(Q K^T / sqrt(d_h) + mask) V.
 *  - same blog, section "CSBP：BP 管损坏块，CP 管干净上下文": forward
 *    O_b = Attn(Q_b, [K_b; K^clean_<b], [V_b; V^clean_<b]); corrupted dQ/dK/dV
 *    stay with the block owner, clean dK/dV accumulate to the clean-shard owner.
 *  - same blog, section "在线 softmax 合并：为什么分两段算仍是同一个注意力":
 *    partial outputs over disjoint key sets merge exactly by log-sum-exp.
 *  - same blog, section "负载均衡：为什么要首尾块配对", and the Turbo-dLLM project
 *    page "Block Parallelism for Efficient Distributed Long-Context Diffusion
 *    Language Model Training", section "Load balancing: pairing early and late
 *    blocks": block b and block B+1-b share a rank; the clean sequence is
 *    sharded with the same early/late (zigzag) pairing.
 * Readings where the pages are silent: clean queries attend block-causally
 * over the clean copy and never read corrupted keys; query head h uses KV
 * head h / (Hq/Hkv); LSE is the natural log of the softmax denominator.
 *
 * Conventions for every entry point:
 *  - Memory is owned by the caller.  The library never allocates or frees
 *    device memory and keeps no state across calls except a per-process
 *    cache of the driver entry point used to encode TMA descriptors.
 *  - Device work is enqueued asynchronously on `stream` (a cudaStream_t
 *    passed as void*; NULL = legacy default stream).  Pointers named *_dev
 *    or documented as "device" must be device (or managed) memory of the
 *    current CUDA device.
 *  - Tensors are bf16, contiguous, layout [batch][L][heads][d] unless stated
 *    (the inputs of csbp_inputs may have token and batch strides).
 *    Every device pointer must be 16-byte aligned.
 *  - Errors are reported only as csbp_status values; arguments are validated
 *    before anything is enqueued, so an error return enqueues no work.  A
 *    device-side wait that exceeds its time budget (a hang guard, never
 *    expected) makes the kernel drain and return; csbp_check_status reports
 *    it afterwards as CSBP_ERR_TIMEOUT.
 */
#ifndef CSBP_H_
#define CSBP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSBP_OK = 0,
  CSBP_ERR_INVALID = -1,     /* bad argument (null, shape, alignment)        */
  CSBP_ERR_UNSUPPORTED = -2, /* valid problem the kernels do not cover       */
  CSBP_ERR_WORKSPACE = -3,   /* workspace smaller than csbp_workspace_bytes  */
  CSBP_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed            */
  CSBP_ERR_TIMEOUT = -5,     /* a bounded device wait gave up                */
  CSBP_ERR_CAPACITY = -6,    /* output buffer too small; size reported       */
  CSBP_ERR_DEVICE = -7       /* a kernel refused its launch environment
                                (shared-memory window not 1024-byte aligned) */
} csbp_status;

/* Problem description.
 *  L      clean length = corrupted length (positions per copy), L % M == 0
 *  M      block size (B = L / M blocks)
 *  Hq,Hkv query / key-value heads, Hq % Hkv == 0 (GQA group G = Hq / Hkv)
 *  d      head dimension: 64 or 128
 *  P      virtual clean shards: 1 = unsharded fused path; P > 1 = one partial
 *         per clean shard plus the corrupted own-block partial, LSE-merged.
 *         P > 1 needs (L/M) % (2P) == 0 and (L/(2P)) % tile_kv == 0.
 *  tile_q, tile_kv  schedule granularity; the kernels need 128 / 128.
 *  has_clean_queries  1 = both copies query; 0 = corrupted queries only
 *         (drafter workload; clean K/V are context only).
 *  scale  softmax scale (1/sqrt(d) for the standard layer).            */
typedef struct {
  int32_t batch, L, M, Hq, Hkv, d, P;
  int32_t tile_q, tile_kv;
  int32_t has_clean_queries;
  float scale;
  int32_t window;       /* 0: none; W > 0: a query reads only keys less than W
                           positions back (i - j < W, positions within each
                           copy), on top of the block rules (sliding-window
                           layers, [Blog] "实验数字：256K 上下文下的主结果")      */
  int32_t clean_causal; /* 0: clean queries block-causal over the clean copy;
                           1: token-causal (key j <= query i)             */
  int32_t bwd_chunk;    /* backward query-tile window, >= 0 (0: none).
                           When a key tile can be read by more query tiles
                           than this, every backward task covers one window
                           of query tiles counted from the last tile, the
                           CTAs of a wave walk the same window, and dK/dV
                           gather in fp32 workspace accumulators (then
                           bf16).  A schedule setting: results differ only
                           by fp32 summation order.                      */
  int32_t per_rank;     /* 0: every query row of the sequence (one GPU runs
                           all P clean shards).  1: only the query rows that
                           CSBP rank `rank` of P > 1 ranks owns -- the clean
                           rows of its two chunks (rank and 2P-1-rank) and
                           the corrupted rows of the blocks inside them --
                           as one rank of a multi-GPU job runs them after
                           the all-gather of the clean K/V shards ([Blog]
                           "在线 softmax 合并：为什么分两段算仍是同一个注意力",
                           implementation schedule).  The clean K/V inputs
                           must then hold the whole clean copy; corrupted
                           K/V rows and query rows the rank does not own are
                           never read.  The forward is one fused pass over
                           the owned query tiles (no partials, no merge) and
                           writes O and LSE of the owned rows only.  The
                           backward writes dQ of the owned rows (other rows
                           zero), dK/dV of the owned corrupted blocks (other
                           corrupted rows zero), and, for every clean key,
                           the part of its dK/dV that the owned query rows
                           contribute: the rank's addend of the owner
                           reduce-scatter.                               */
  int32_t rank;         /* 0 <= rank < P when per_rank == 1, else 0       */
} csbp_problem;

/* Device input tensors, bf16 [batch][L][H][d] (H = Hq for q, Hkv for k/v).
 * q_clean may be NULL when has_clean_queries == 0.
 *
 * Within a token the H heads of d features are contiguous (head stride d).
 * Tokens and batch entries may be strided, so q, k and v can be views into
 * one packed projection output, [batch][L][Hq + 2 Hkv][d] for example.
 * stride_tok[i] and stride_batch[i] are element strides for the i-th
 * pointer above (order q_clean, k_clean, v_clean, q_corr, k_corr, v_corr):
 *   stride_tok[i]    0 = H*d (contiguous); else >= H*d and a multiple of 8;
 *   stride_batch[i]  0 = L*stride_tok[i]; else >= L*stride_tok[i] and a
 *                    multiple of 8; read only when batch > 1.
 * Both must stay below 2^39 elements, and every pointer is 16-byte aligned.
 * A zero-initialised struct with the six pointers set is the contiguous
 * layout.  A stride outside these rules gives CSBP_ERR_INVALID.           */
typedef struct {
  const void *q_clean, *k_clean, *v_clean;
  const void *q_corr, *k_corr, *v_corr;
  int64_t stride_tok[6];
  int64_t stride_batch[6];
} csbp_inputs;

/* Summary of a work list built by csbp_block_schedule. */
typedef struct {
  int32_t n_fwd_tasks;    /* forward tasks (one query tile [x part])      */
  int32_t n_fwd_segments; /* key-tile ranges of the forward tasks         */
  int32_t n_bwd_tasks;    /* backward tasks (one key tile)                */
  int32_t n_bwd_segments; /* query-tile ranges of the backward tasks      */
  int64_t tile_pairs;     /* (query tile, key tile) pairs with >=1 allowed entry */
  int64_t bytes;          /* size of the work list                        */
  uint64_t problem_key;   /* opaque fingerprint of the problem fields the
                             list depends on (L, M, tiles, P, query copies,
                             window, clean_causal, bwd_chunk, per_rank,
                             rank); the attention
                             entry points refuse, with CSBP_ERR_INVALID, an
                             info whose key does not match their problem   */
} csbp_schedule_info;

/* Work-list layout (int32 words; produced and consumed only by this library
 * but documented for tests):
 *   words[0..15]  header: magic 0x43534250, version 1, L, M, tile, P,
 *                 has_clean_queries, n_fwd_tasks, n_fwd_segments,
 *                 n_bwd_tasks, n_bwd_segments, off_fwd_tasks, off_fwd_segs,
 *                 off_bwd_tasks, off_bwd_segs, total_words
 *   fwd task (8 words): q_stream, q_tile, part (-1 = all parts, fused),
 *                 seg_begin, seg_count, kv_tiles, 0, 0
 *   fwd segment (4 words): kv_stream, kv_tile_begin, kv_tile_end (exclusive),
 *                 flags (bit0 = partial: tiles need the in-tile mask)
 *   bwd task (8 words): kv_stream, kv_tile, part, seg_begin, seg_count,
 *                 q_tiles, flags (bit0 = dK/dV add into the fp32
 *                 accumulators), window (0 = the last bwd_chunk query
 *                 tiles, 1 = the ones before, ...).  One task per key tile
 *                 of both copies, including tiles no query reads (dK/dV
 *                 zero); with windows, one per key tile and window that
 *                 holds a query tile reading it.
 *   bwd segment (4 words): q_stream, q_tile_begin, q_tile_end, flags
 * Streams: 0 = clean copy, 1 = corrupted copy.  Part of a key tile: the
 * owner shard of its clean chunk (clean keys) or P (corrupted keys).
 * Tasks are ordered heaviest first (ties in canonical order).            */

/* Build the dual-end block ownership, the zigzag clean-chunk ownership and
 * the mask-aware tile work list on the host (no CUDA call).
 *  block_owner  host int32[B] or NULL: owner shard of each corrupted block
 *  chunk_owner  host int32[2P] or NULL: owner shard of each clean chunk
 *  work         host buffer for the work list, or NULL to query the size
 *  work_cap     capacity of `work` in bytes
 *  info         out: counts, the required size in bytes and the problem
 *               fingerprint (always filled on CSBP_OK and CSBP_ERR_CAPACITY);
 *               pass it with the list to csbp_attn_fwd / csbp_attn_bwd
 * Shard r owns clean chunks r and 2P-1-r of the 2P contiguous chunks of
 * length L/(2P); a corrupted block is owned by the owner of the chunk that
 * holds its first position (so blocks b and B-1-b pair up, 0-based).
 * Returns CSBP_ERR_CAPACITY if work is NULL or too small.               */
csbp_status csbp_block_schedule(const csbp_problem* problem, int32_t* block_owner,
                                int32_t* chunk_owner, void* work, int64_t work_cap,
                                csbp_schedule_info* info);

/* Bytes of device workspace needed: which = 0 forward, 1 backward.
 * Forward: a status word, plus for P > 1 the fp32 partials
 *   (P+1) x 2 x batch x L x Hq x (d + 1) x 4 bytes.
 * Backward: a status word, D (2 x batch x Hq x L fp32) and the fp32 dQ
 *   accumulator (2 x batch x L x Hq x d).  Returns 0 for an invalid problem. */
size_t csbp_workspace_bytes(const csbp_problem* problem, int which);

/* Forward.  work_dev: device copy of the work list from csbp_block_schedule
 * for this problem (info: its summary).  Outputs (device):
 *   o_clean, o_corr  bf16 [batch][L][Hq][d]  (o_clean ignored, may be NULL,
 *                    when has_clean_queries == 0)
 *   lse              fp32 [batch][2][Hq][L], natural-log softmax denominator
 *                    of each query row (copy 0 untouched without clean queries)
 * P == 1: one fused pass per query tile over all its allowed key tiles.
 * P > 1: per-part partial attention into the workspace, then the LSE merge.
 * workspace: device, >= csbp_workspace_bytes(problem, 0); its first 256
 * bytes (the status word) zeroed before its first use (csbp_check_status). */
csbp_status csbp_attn_fwd(const csbp_problem* problem, const csbp_inputs* in,
                          const void* work_dev, const csbp_schedule_info* info,
                          void* o_clean, void* o_corr, float* lse, void* workspace,
                          size_t ws_bytes, void* stream);

/* Backward (exact): given the forward's O and LSE and the upstream dO,
 * writes dQ for each query copy and dK, dV for each key copy (bf16, same
 * layouts as the inputs; dK/dV summed over the G query heads of each KV
 * head; outputs are overwritten, not accumulated).  Clean dK/dV collect
 * contributions from clean queries of the same or later blocks and from
 * corrupted queries of later blocks; corrupted dK/dV only from queries of
 * their own block.  do_clean / dq_clean may be NULL without clean queries.
 * Needs L % 4 == 0 (the LSE and D rows are TMA-loaded), else
 * CSBP_ERR_UNSUPPORTED.
 * workspace: device, >= csbp_workspace_bytes(problem, 1); its first 256
 * bytes (the status word) zeroed before its first use (csbp_check_status). */
csbp_status csbp_attn_bwd(const csbp_problem* problem, const csbp_inputs* in,
                          const void* work_dev, const csbp_schedule_info* info,
                          const void* o_clean, const void* o_corr, const float* lse,
                          const void* do_clean, const void* do_corr, void* dq_clean,
                          void* dq_corr, void* dk_clean, void* dv_clean, void* dk_corr,
                          void* dv_corr, void* workspace, size_t ws_bytes, void* stream);

/* Backward without any workspace argument, for callers that cannot allocate
 * device memory (plugin or custom-op interfaces that receive only their
 * input and output buffers, runtimes whose memory pool forbids outside
 * allocations, paths that cannot afford cudaMalloc's implicit device
 * synchronisation).  This entry point has no counterpart on the method's
 * pages; it is a deployment convenience of this library.
 * Same arguments, layouts and results as csbp_attn_bwd, minus the
 * workspace.  Its scratch is one fixed 64 MiB array in device global memory
 * that every GPU loading the library holds until the process exits; a
 * problem whose csbp_workspace_bytes(problem, 1) exceeds 64 MiB is rejected
 * with CSBP_ERR_WORKSPACE before anything is enqueued.  It allocates and
 * frees nothing.  The first call on a device looks up the array's device
 * address (make that first call before any stream capture).  All calls on a
 * device share the array and it keeps the last call's contents: each call
 * clears the part that must start at zero, and calls that can overlap on the
 * GPU (for example on two streams without ordering) race and corrupt each
 * other's results.  The array's address is cached per device and CUDA
 * context (another context of the device, made current through the driver
 * API, looks it up again); after cudaDeviceReset the device's code is
 * reloaded, so a process that resets a device must not call this entry
 * point on it again.  A device wait that timed out is reported by
 * csbp_attn_bwd_noalloc_status; each call clears the status word first, so
 * check it after the call whose result matters.                          */
csbp_status csbp_attn_bwd_noalloc(const csbp_problem* problem, const csbp_inputs* in,
                                  const void* work_dev, const csbp_schedule_info* info,
                                  const void* o_clean, const void* o_corr, const float* lse,
                                  const void* do_clean, const void* do_corr, void* dq_clean,
                                  void* dq_corr, void* dk_clean, void* dv_clean, void* dk_corr,
                                  void* dv_corr, void* stream);

/* Status of the last csbp_attn_bwd_noalloc call(s) on the current device:
 * synchronises `stream`, then reads and clears the status word at the start
 * of the built-in scratch array, with the codes of csbp_check_status
 * (CSBP_ERR_TIMEOUT if a bounded device wait gave up).  It allocates
 * nothing.  No counterpart on the method's pages.                        */
csbp_status csbp_attn_bwd_noalloc_status(void* stream);

/* Exact log-sum-exp merge of n_parts partial attentions over disjoint key
 * sets (blog section "在线 softmax 合并"): m = max_s z_s, w_s = exp(z_s - m),
 * O = sum_s w_s O_s / sum_s w_s, z = m + log(sum_s w_s), all in fp32; a part
 * with z = -inf read no key and has weight 0.
 *  o_parts   host array of n_parts device pointers, fp32 [rows][Hq][d]
 *  lse_parts host array of n_parts device pointers, fp32 [Hq][rows]
 *  o_out     device bf16 [rows][Hq][d];  lse_out device fp32 [Hq][rows]
 * 1 <= n_parts <= 64, d % 4 == 0, rows x Hq x d < 2^39.  Alignment: the
 * o_parts 16 bytes, o_out 16 bytes (8 when d % 8 == 0), the LSE arrays 4
 * bytes; anything else gives CSBP_ERR_INVALID before a launch.           */
csbp_status csbp_lse_merge(int32_t n_parts, const float* const* o_parts,
                           const float* const* lse_parts, int64_t rows, int32_t Hq,
                           int32_t d, void* o_out, float* lse_out, void* stream);

/* fp8 inputs.  Decodes n bytes of OCP 8-bit floating point, variant E4M3
 * (sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
 * subnormal; no infinities; S.1111.111 is NaN) and writes, in bf16,
 *   out[i] = bf16_rn(fp32(scale * value(in[i])))
 * -- one fp32 multiply (exact when scale is a power of two) rounded to bf16,
 * nearest even; NaN stays NaN.  For Q, K, V and dO kept in fp8 with one scale
 * per tensor: decode them into bf16 buffers and call the attention entry
 * points, whose arithmetic is unchanged (bf16 operands, fp32 accumulation).
 * The method's pages fix no precision; this is the fp8-input workload.
 *  in   device, n bytes;  out  device, n bf16 elements; both 16-byte aligned
 *  0 <= n < 2^40; scale finite and nonzero, else CSBP_ERR_INVALID.       */
csbp_status csbp_e4m3_to_bf16(const void* in, float scale, void* out, int64_t n, void* stream);

/* Synchronise `stream`, then read and clear the device status word kept at
 * the start of `workspace` by csbp_attn_fwd / csbp_attn_bwd.  The entry
 * points only ever set that word (the first 256 bytes of a workspace), so
 * a caller zeroes it once, before the first call with a fresh workspace
 * (cudaMemset); from then on this function clears it after each read.  Returns
 * CSBP_ERR_TIMEOUT if a bounded device wait gave up since the last check,
 * CSBP_ERR_DEVICE if a kernel refused to run: its shared-memory window was
 * not 1024-byte aligned, or (debug build, libcsbp_debug.so) a work-list
 * record it was given points outside the list or the sequence; such a CTA
 * writes nothing. */
csbp_status csbp_check_status(void* workspace, void* stream);

/* Kernel timing, a profiling aid with no counterpart in the method; off by
 * default.  csbp_kernel_timing(1) creates a pool of CUDA events on the
 * current device and clears the record; while it is on, every csbp_attn_fwd
 * and csbp_attn_bwd call records an event pair on its stream around its main
 * kernel (fwd_kernel / bwd_kernel) and its HBM-bound launches, and
 * csbp_vocab_ce one around each of its launches, up to 4096 pairs in all
 * (later launches are not timed).
 * csbp_kernel_timing(0) stops recording and keeps the record.
 * csbp_kernel_timing_read synchronises the recorded events and returns the
 * summed device milliseconds and launch counts of each kind (any output
 * pointer may be NULL).  CSBP_ERR_CUDA if an event call fails. */
csbp_status csbp_kernel_timing(int32_t enable);
csbp_status csbp_kernel_timing_read(double* fwd_ms, int32_t* n_fwd, double* bwd_ms,
                                    int32_t* n_bwd);

/* The same record by kernel kind: 0 fwd_kernel, 1 bwd_kernel; for
 * csbp_vocab_ce (csbp_vocab_ce.h) 2 the logits GEMM, 3 the row kernel
 * (LSE, loss, g), 4 the dH GEMM, 5 the dW GEMM; and the HBM-bound launches
 * of the attention calls: 6 the LSE merge (one per query stream and batch
 * entry), 7 the backward preprocess and 8 the dQ convert (one per query
 * stream), 9 the dK/dV converts of a windowed backward (one pair per key
 * stream); 10 csbp_e4m3_to_bf16.  One event pair per launch.
 * CSBP_ERR_INVALID for another kind. */
csbp_status csbp_kernel_timing_read_kind(int32_t kind, double* ms, int32_t* n);

/* Self-test of the device hang guard: launches one small kernel on `stream`
 * that waits, through the kernels' bounded-wait helpers, on a barrier that
 * nothing ever arrives on; after budget_ns (1e3 .. 2e9) of wall time the
 * wait gives up and records a timeout in the status word at the start of
 * `workspace` (>= 256 bytes, 16-byte aligned, device memory), exactly as a
 * hung attention or GEMM kernel would.  csbp_check_status then returns
 * CSBP_ERR_TIMEOUT (and clears the word); nothing else is left in flight, so
 * the context stays usable.  CSBP_ERR_INVALID for a bad argument. */
csbp_status csbp_wait_selftest(int64_t budget_ns, void* workspace, void* stream);

/* Human-readable name of a status code (static string). */
const char* csbp_status_string(csbp_status status);

/* Library version: major * 10000 + minor * 100 + patch.  0.2.0 (200) added
 * csbp_problem.window / clean_causal / bwd_chunk, csbp_vocab_ce (with
 * csbp_vocab_ce.h), csbp_wait_selftest and csbp_kernel_timing_read_kind.
 * 0.3.0 (300) added the token and batch strides of csbp_inputs and
 * csbp_schedule_info.problem_key.  0.4.0 (400) added csbp_problem.per_rank
 * and rank (one CSBP rank's query rows) and csbp_attn_bwd_noalloc_status. */
int32_t csbp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSBP_H_ */
