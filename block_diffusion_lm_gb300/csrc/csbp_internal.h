// Internal declarations shared by the translation units of libcsbp.
#pragma once

#include <cstdint>

#include "csbp.h"

namespace csbp {

constexpr int32_t kMagic = 0x43534250;  // 'CSBP'
constexpr int32_t kVersion = 1;
constexpr int kHeaderWords = 16;
constexpr int kTaskWords = 8;
constexpr int kSegWords = 4;
constexpr int kMaxParts = 64;
constexpr int kTile = 128;  // query and key tile rows of the kernels

// Header word indices of a work list.
enum HeaderWord {
  H_MAGIC = 0, H_VERSION, H_L, H_M, H_TILE, H_P, H_HAS_CLEAN, H_N_FWD_TASKS,
  H_N_FWD_SEGS, H_N_BWD_TASKS, H_N_BWD_SEGS, H_OFF_FWD_TASKS, H_OFF_FWD_SEGS,
  H_OFF_BWD_TASKS, H_OFF_BWD_SEGS, H_TOTAL
};

csbp_status validate_problem(const csbp_problem* p);

// Backward query-tile window (csbp_problem::bwd_chunk) and whether the
// problem's backward runs in windows with fp32 dK/dV accumulation: only on
// request (bwd_chunk > 0), once a key tile can be read by more query tiles
// than that.  With the KV-head-major CTA order long sequences measured
// faster without windows (a 1M-token corrupted-only backward: 1080 vs 1017
// TFLOP/s), so the default never windows.
int64_t bwd_chunk_tiles(const csbp_problem* p);
bool bwd_windowed(const csbp_problem* p);

// Kernel timing (csbp_kernel_timing): kinds 0 fwd, 1 bwd, 2 CE logits GEMM,
// 3 CE row kernel, 4 CE dH GEMM, 5 CE dW GEMM, 6 LSE merge, 7 backward
// preprocess, 8 dQ convert, 9 dK/dV convert (windowed backward), 10 fp8
// E4M3 input decode.
// timer_begin returns the pair index to close with timer_end, or -1 when not
// recording.
constexpr int kTimerKinds = 11;
int timer_begin(int kind, void* stream);
void timer_end(int i, void* stream);

// Encode a 2-D TMA descriptor (a CUtensorMap at `map`) over a row-major
// array of `outer` rows of `inner` elements (bf16, or fp32 if `f32`), rows
// `row_bytes` apart; box = box_inner x box_outer elements, 128-byte swizzle
// if `swizzle128`; out-of-range elements read as zero.
bool encode_map_2d(void* map, bool f32, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);
int classify_tile(int q_stream, int64_t qt, int k_stream, int64_t kt, int64_t L, int64_t M,
                  int64_t T);

// Launch-side parameter blocks (plain data, passed by value to kernels).
struct FwdParams {
  const int32_t* tasks;  // device: fwd task records
  const int32_t* segs;   // device: fwd segment records
  int32_t L, M, Hq, Hkv, G, batch;
  int32_t window, clean_causal;  // mask options (0 = none / block-causal)
  int32_t n_segs, nT;    // segment records, tiles per copy (debug-build checks)
  float scale_log2;      // softmax scale * log2(e)
  void* o[2];            // bf16 outputs per query stream
  float* lse;            // [batch][2][Hq][L]
  float* part_o;         // [(P+1)][2][batch][L][Hq][d] fp32 (partial mode)
  float* part_lse;       // [(P+1)][2][batch][Hq][L]
  int32_t partial_mode;
  int* status;
};

// Per-part pointers of one LSE merge (o: [rows][Hq][d] fp32, z: [Hq][rows]).
struct MergeArgs {
  const float* o[kMaxParts];
  const float* z[kMaxParts];
};

struct BwdParams {
  const int32_t* tasks;  // device: bwd task records
  const int32_t* segs;   // device: bwd segment records
  int32_t L, M, Hq, Hkv, G, batch;
  int32_t window, clean_causal;  // mask options (0 = none / block-causal)
  int32_t n_segs, nT;    // segment records, tiles per copy (debug-build checks)
  float scale_log2;
  float scale;
  float* dq_acc;         // [2][batch][L][Hq][d] fp32, pre-zeroed
  void* dk[2];           // bf16 [batch][L][Hkv][d] per key stream
  void* dv[2];
  float* dk_acc;         // windowed backward: fp32 [2][batch][L][Hkv][d], pre-zeroed
  float* dv_acc;
  int32_t kv_major;      // CTA order: 1 = (batch, KV head) outer, task inner
  int* status;
};

}  // namespace csbp
