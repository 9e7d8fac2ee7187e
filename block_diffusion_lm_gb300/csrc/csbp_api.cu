// C-ABI entry points of libcsbp: argument validation, TMA descriptor
// encoding, workspace carving and kernel launches.  No entry point allocates
// memory; all device work goes to the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "csbp.h"
#include "csbp_internal.h"

namespace csbp {

cudaError_t launch_fwd(int d, const CUtensorMap* maps, const FwdParams& p, int n_tasks,
                       cudaStream_t stream);
cudaError_t launch_bwd(int d, const CUtensorMap* maps, const BwdParams& p, int n_tasks,
                       cudaStream_t stream);
int bwd_query_box_rows();
int bwd_dq_box_rows(int d);
cudaError_t launch_lse_merge(const MergeArgs& a, int n_parts, int64_t rows, int Hq, int d,
                             void* o_out, float* z_out, cudaStream_t stream);
cudaError_t launch_bwd_pre(int d, const void* o, const void* dO, float* Dsum, float* dq_acc,
                           int64_t rows, int Hq, int L, cudaStream_t stream);
cudaError_t launch_dq_convert(const float* acc, void* dq, int64_t n_elems, float scale,
                              cudaStream_t stream);
cudaError_t launch_fill(float* x, int64_t n, float v, cudaStream_t stream);
cudaError_t launch_e4m3_to_bf16(const void* in, void* out, int64_t n, float scale,
                                cudaStream_t stream);
uint64_t schedule_key(const csbp_problem* p);

namespace {

constexpr size_t kStatusBytes = 256;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a bf16 [batch][L][H][d] tensor viewed as {H*d, L, batch};
// box = 64 elements (128 B, one swizzle row) x box_rows rows x 1.
// Element strides of one bf16 [batch][L][H][d] tensor between tokens and
// between batch entries (heads and features are always contiguous).
struct TokStride {
  int64_t tok, batch;
};

TokStride contiguous_stride(int64_t H, int d, int64_t L) {
  return {H * d, L * H * d};
}

// Strides of the i-th pointer of csbp_inputs (q_clean, k_clean, v_clean,
// q_corr, k_corr, v_corr): the caller's, or the contiguous ones for 0.
TokStride input_stride(const csbp_problem* p, const csbp_inputs* in, int i) {
  const int64_t H = (i == 0 || i == 3) ? p->Hq : p->Hkv;
  TokStride s;
  s.tok = in->stride_tok[i] != 0 ? in->stride_tok[i] : H * p->d;
  s.batch = (p->batch > 1 && in->stride_batch[i] != 0) ? in->stride_batch[i]
                                                        : static_cast<int64_t>(p->L) * s.tok;
  return s;
}

// 3-D map {H*d, L, batch} over a bf16 [batch][L][H][d] tensor with the given
// token and batch strides; box = 64 features x box_rows tokens x 1.
bool make_map(CUtensorMap* m, const void* base, int64_t H, int d, int64_t L, int64_t batch,
              TokStride st, int box_rows = kTile) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(H * d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(st.tok * 2),
                           static_cast<cuuint64_t>(st.batch * 2)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over an fp32 [rows][L] array; box = box_len consecutive positions
// of one row (positions >= L read as zero).  Needs L % 4 == 0 (16-byte rows).
bool make_map_rows_f32(CUtensorMap* m, const void* base, int64_t L, int64_t rows, int box_len) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(L * 4)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_len), 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the fp32 dQ accumulator [2*batch][L][Hq][d] viewed as
// {Hq*d, L, 2*batch}; box = d elements x box_rows rows x 1, no swizzle (the
// target of the backward's TMA reduce-adds; rows >= L are clipped).
bool make_map_dqacc(CUtensorMap* m, void* base, int64_t Hq, int d, int64_t L, int64_t planes,
                    int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(Hq * d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(Hq * d * 4),
                           static_cast<cuuint64_t>(L * Hq * d * 4)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct WsLayout {
  size_t status = 0, part_o = 0, part_lse = 0, dsum = 0, dq_acc = 0, dk_acc = 0, dv_acc = 0,
         total = 0;
};

WsLayout ws_layout(const csbp_problem* p, int which) {
  WsLayout w;
  const size_t rows = static_cast<size_t>(p->batch) * p->L;
  size_t off = kStatusBytes;
  if (which == 0) {
    if (p->P > 1 && !p->per_rank) {  // a rank's forward is one fused pass
      w.part_o = off;
      off += round256(static_cast<size_t>(p->P + 1) * 2 * rows * p->Hq * p->d * 4);
      w.part_lse = off;
      off += round256(static_cast<size_t>(p->P + 1) * 2 * rows * p->Hq * 4);
    }
  } else {
    w.dsum = off;
    off += round256(2 * rows * p->Hq * 4);
    w.dq_acc = off;
    off += round256(2 * rows * p->Hq * p->d * 4);
    if (bwd_windowed(p)) {
      w.dk_acc = off;
      off += round256(2 * rows * p->Hkv * p->d * 4);
      w.dv_acc = off;
      off += round256(2 * rows * p->Hkv * p->d * 4);
    }
  }
  w.total = off;
  return w;
}

csbp_status check_inputs(const csbp_problem* p, const csbp_inputs* in) {
  if (!in) return CSBP_ERR_INVALID;
  if (!in->k_clean || !in->v_clean || !in->q_corr || !in->k_corr || !in->v_corr)
    return CSBP_ERR_INVALID;
  if (p->has_clean_queries && !in->q_clean) return CSBP_ERR_INVALID;
  const void* ptrs[6] = {in->q_clean, in->k_clean, in->v_clean, in->q_corr, in->k_corr, in->v_corr};
  constexpr int64_t kMaxStride = int64_t(1) << 39;  // elements: TMA strides stay below 2^40 bytes
  for (int i = 0; i < 6; ++i) {
    if (!ptrs[i]) continue;
    if (!aligned16(ptrs[i])) return CSBP_ERR_INVALID;
    if (in->stride_tok[i] < 0 || in->stride_batch[i] < 0) return CSBP_ERR_INVALID;
    const int64_t H = (i == 0 || i == 3) ? p->Hq : p->Hkv;
    // 16-byte rows for TMA; one batch entry (L tokens) below 2^39 elements,
    // tested by division so that no product can overflow
    const int64_t tok = in->stride_tok[i] != 0 ? in->stride_tok[i] : H * p->d;
    if (tok < H * p->d || tok % 8 != 0 || tok > (kMaxStride - 1) / p->L) return CSBP_ERR_INVALID;
    const TokStride s = input_stride(p, in, i);
    // batch entries that do not overlap
    if (s.batch < static_cast<int64_t>(p->L) * s.tok || s.batch % 8 != 0 ||
        s.batch >= kMaxStride)
      return CSBP_ERR_INVALID;
  }
  return CSBP_OK;
}

// Offsets of the four record arrays, from the deterministic layout.
struct WorkOffsets {
  int64_t fwd_tasks, fwd_segs, bwd_tasks, bwd_segs;
};

WorkOffsets work_offsets(const csbp_schedule_info* info) {
  WorkOffsets o;
  o.fwd_tasks = kHeaderWords;
  o.fwd_segs = o.fwd_tasks + static_cast<int64_t>(info->n_fwd_tasks) * kTaskWords;
  o.bwd_tasks = o.fwd_segs + static_cast<int64_t>(info->n_fwd_segments) * kSegWords;
  o.bwd_segs = o.bwd_tasks + static_cast<int64_t>(info->n_bwd_tasks) * kTaskWords;
  return o;
}

// ---------------------------------------------------------------- timing
// Event pairs around the main kernels, for csbp_kernel_timing(_read).
struct KernelTimer {
  static constexpr int kCap = 4096;
  std::mutex mu;
  bool on = false;
  int device = -1;
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> kind;  // timer kind of each recorded pair (see csbp.h)
};
KernelTimer& timer() {
  static KernelTimer t;
  return t;
}

}  // namespace

int timer_begin(int kind, void* stream) {
  KernelTimer& t = timer();
  std::lock_guard<std::mutex> lk(t.mu);
  if (!t.on || static_cast<int>(t.kind.size()) >= KernelTimer::kCap) return -1;
  const int i = static_cast<int>(t.kind.size());
  if (cudaEventRecord(t.start[i], static_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  t.kind.push_back(kind);
  return i;
}

void timer_end(int i, void* stream) {
  if (i < 0) return;
  KernelTimer& t = timer();
  std::lock_guard<std::mutex> lk(t.mu);
  cudaEventRecord(t.stop[i], static_cast<cudaStream_t>(stream));
}

bool encode_map_2d(void* map, bool f32, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(static_cast<CUtensorMap*>(map),
                   f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace csbp

using namespace csbp;

extern "C" csbp_status csbp_kernel_timing(int32_t enable) {
  KernelTimer& t = timer();
  std::lock_guard<std::mutex> lk(t.mu);
  if (!enable) {
    t.on = false;
    return CSBP_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSBP_ERR_CUDA;
  if (t.device != dev) {
    for (auto e : t.start) cudaEventDestroy(e);
    for (auto e : t.stop) cudaEventDestroy(e);
    t.start.assign(KernelTimer::kCap, nullptr);
    t.stop.assign(KernelTimer::kCap, nullptr);
    for (int i = 0; i < KernelTimer::kCap; ++i) {
      if (cudaEventCreate(&t.start[i]) != cudaSuccess || cudaEventCreate(&t.stop[i]) != cudaSuccess) {
        t.device = -1;
        return CSBP_ERR_CUDA;
      }
    }
    t.device = dev;
  }
  t.kind.clear();
  t.on = true;
  return CSBP_OK;
}

extern "C" csbp_status csbp_kernel_timing_read(double* fwd_ms, int32_t* n_fwd, double* bwd_ms,
                                               int32_t* n_bwd) {
  KernelTimer& t = timer();
  std::lock_guard<std::mutex> lk(t.mu);
  double ms[2] = {0.0, 0.0};
  int32_t n[2] = {0, 0};
  for (size_t i = 0; i < t.kind.size(); ++i) {
    if (t.kind[i] > 1) continue;
    float e = 0.f;
    if (cudaEventSynchronize(t.stop[i]) != cudaSuccess ||
        cudaEventElapsedTime(&e, t.start[i], t.stop[i]) != cudaSuccess)
      return CSBP_ERR_CUDA;
    ms[t.kind[i]] += e;
    n[t.kind[i]] += 1;
  }
  if (fwd_ms) *fwd_ms = ms[0];
  if (n_fwd) *n_fwd = n[0];
  if (bwd_ms) *bwd_ms = ms[1];
  if (n_bwd) *n_bwd = n[1];
  return CSBP_OK;
}

extern "C" csbp_status csbp_kernel_timing_read_kind(int32_t kind, double* ms, int32_t* n) {
  if (kind < 0 || kind >= kTimerKinds) return CSBP_ERR_INVALID;
  KernelTimer& t = timer();
  std::lock_guard<std::mutex> lk(t.mu);
  double sum = 0.0;
  int32_t cnt = 0;
  for (size_t i = 0; i < t.kind.size(); ++i) {
    if (t.kind[i] != kind) continue;
    float e = 0.f;
    if (cudaEventSynchronize(t.stop[i]) != cudaSuccess ||
        cudaEventElapsedTime(&e, t.start[i], t.stop[i]) != cudaSuccess)
      return CSBP_ERR_CUDA;
    sum += e;
    ++cnt;
  }
  if (ms) *ms = sum;
  if (n) *n = cnt;
  return CSBP_OK;
}

extern "C" int32_t csbp_version(void) { return 400; }  // 0.4.0: per-rank query rows

extern "C" const char* csbp_status_string(csbp_status s) {
  switch (s) {
    case CSBP_OK: return "ok";
    case CSBP_ERR_INVALID: return "invalid argument";
    case CSBP_ERR_UNSUPPORTED: return "unsupported problem";
    case CSBP_ERR_WORKSPACE: return "workspace too small";
    case CSBP_ERR_CUDA: return "CUDA error";
    case CSBP_ERR_TIMEOUT: return "device wait timed out";
    case CSBP_ERR_CAPACITY: return "output buffer too small";
    case CSBP_ERR_DEVICE: return "kernel refused its launch environment";
  }
  return "unknown status";
}

extern "C" size_t csbp_workspace_bytes(const csbp_problem* problem, int which) {
  if (validate_problem(problem) != CSBP_OK || (which != 0 && which != 1)) return 0;
  return ws_layout(problem, which).total;
}

extern "C" csbp_status csbp_attn_fwd(const csbp_problem* problem, const csbp_inputs* in,
                                     const void* work_dev, const csbp_schedule_info* info,
                                     void* o_clean, void* o_corr, float* lse, void* workspace,
                                     size_t ws_bytes, void* stream_) {
  csbp_status st = validate_problem(problem);
  if (st != CSBP_OK) return st;
  if (problem->tile_q != kTile) return CSBP_ERR_UNSUPPORTED;
  if ((st = check_inputs(problem, in)) != CSBP_OK) return st;
  if (!work_dev || !info || !o_corr || !lse || !workspace) return CSBP_ERR_INVALID;
  if (info->problem_key != schedule_key(problem)) return CSBP_ERR_INVALID;  // another problem's list
  if (problem->has_clean_queries && !o_clean) return CSBP_ERR_INVALID;
  if (!aligned16(work_dev) || !aligned16(o_corr) || (o_clean && !aligned16(o_clean)) ||
      !aligned16(lse) || !aligned16(workspace))
    return CSBP_ERR_INVALID;
  const WsLayout wl = ws_layout(problem, 0);
  if (ws_bytes < wl.total) return CSBP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const csbp_problem& p = *problem;

  CUtensorMap maps[6];
  const int qi = in->q_clean ? 0 : 3;  // the clean-query map is unused when absent
  const void* qc = in->q_clean ? in->q_clean : in->q_corr;
  if (!make_map(&maps[0], qc, p.Hq, p.d, p.L, p.batch, input_stride(problem, in, qi)) ||
      !make_map(&maps[1], in->q_corr, p.Hq, p.d, p.L, p.batch, input_stride(problem, in, 3)) ||
      !make_map(&maps[2], in->k_clean, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 1)) ||
      !make_map(&maps[3], in->k_corr, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 4)) ||
      !make_map(&maps[4], in->v_clean, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 2)) ||
      !make_map(&maps[5], in->v_corr, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 5)))
    return CSBP_ERR_CUDA;

  const WorkOffsets wo = work_offsets(info);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FwdParams fp;
  fp.tasks = static_cast<const int32_t*>(work_dev) + wo.fwd_tasks;
  fp.segs = static_cast<const int32_t*>(work_dev) + wo.fwd_segs;
  fp.L = p.L;
  fp.M = p.M;
  fp.Hq = p.Hq;
  fp.Hkv = p.Hkv;
  fp.G = p.Hq / p.Hkv;
  fp.batch = p.batch;
  fp.window = p.window;
  fp.clean_causal = p.clean_causal;
  fp.n_segs = info->n_fwd_segments;
  fp.nT = (p.L + kTile - 1) / kTile;
  fp.scale_log2 = p.scale * 1.4426950408889634f;
  fp.o[0] = o_clean;
  fp.o[1] = o_corr;
  fp.lse = lse;
  fp.part_o = nullptr;
  fp.part_lse = nullptr;
  const bool partial = p.P > 1 && !p.per_rank;  // virtual shards: partials + merge
  fp.partial_mode = partial ? 1 : 0;
  fp.status = reinterpret_cast<int*>(ws + wl.status);
  if (partial) {
    fp.part_o = reinterpret_cast<float*>(ws + wl.part_o);
    fp.part_lse = reinterpret_cast<float*>(ws + wl.part_lse);
    const int64_t n_lse = static_cast<int64_t>(p.P + 1) * 2 * p.batch * p.Hq * p.L;
    if (launch_fill(fp.part_lse, n_lse, -INFINITY, stream) != cudaSuccess) return CSBP_ERR_CUDA;
  }
  const int timed = timer_begin(0, stream);
  const cudaError_t fe = launch_fwd(p.d, maps, fp, info->n_fwd_tasks, stream);
  timer_end(timed, stream);
  if (fe != cudaSuccess) return CSBP_ERR_CUDA;
  if (partial) {
    const int n_parts = p.P + 1;
    const int64_t slab_o = static_cast<int64_t>(p.L) * p.Hq * p.d;
    const int64_t slab_z = static_cast<int64_t>(p.Hq) * p.L;
    for (int qs = p.has_clean_queries ? 0 : 1; qs < 2; ++qs) {
      for (int bz = 0; bz < p.batch; ++bz) {
        MergeArgs a;
        for (int s = 0; s < n_parts; ++s) {
          const int64_t prow = (static_cast<int64_t>(s) * 2 + qs) * p.batch + bz;
          a.o[s] = fp.part_o + prow * slab_o;
          a.z[s] = fp.part_lse + prow * slab_z;
        }
        void* oo = static_cast<uint16_t*>(qs ? o_corr : o_clean) + bz * slab_o;  // bf16 elements
        float* zo = lse + (static_cast<int64_t>(bz) * 2 + qs) * slab_z;
        const int tm = timer_begin(6, stream);
        const cudaError_t me = launch_lse_merge(a, n_parts, p.L, p.Hq, p.d, oo, zo, stream);
        timer_end(tm, stream);
        if (me != cudaSuccess)
          return CSBP_ERR_CUDA;
      }
    }
  }
  return CSBP_OK;
}

extern "C" csbp_status csbp_attn_bwd(const csbp_problem* problem, const csbp_inputs* in,
                                     const void* work_dev, const csbp_schedule_info* info,
                                     const void* o_clean, const void* o_corr, const float* lse,
                                     const void* do_clean, const void* do_corr, void* dq_clean,
                                     void* dq_corr, void* dk_clean, void* dv_clean, void* dk_corr,
                                     void* dv_corr, void* workspace, size_t ws_bytes,
                                     void* stream_) {
  csbp_status st = validate_problem(problem);
  if (st != CSBP_OK) return st;
  if (problem->tile_q != kTile) return CSBP_ERR_UNSUPPORTED;
  if (problem->L % 4 != 0) return CSBP_ERR_UNSUPPORTED;  // LSE / D rows are TMA-loaded
  if ((st = check_inputs(problem, in)) != CSBP_OK) return st;
  const bool hc = problem->has_clean_queries != 0;
  if (!work_dev || !info || !o_corr || !lse || !do_corr || !dq_corr || !dk_clean || !dv_clean ||
      !dk_corr || !dv_corr || !workspace)
    return CSBP_ERR_INVALID;
  if (hc && (!o_clean || !do_clean || !dq_clean)) return CSBP_ERR_INVALID;
  if (info->problem_key != schedule_key(problem)) return CSBP_ERR_INVALID;  // another problem's list
  const void* all[] = {work_dev, o_corr, lse, do_corr, dq_corr, dk_clean, dv_clean, dk_corr,
                       dv_corr, workspace, o_clean, do_clean, dq_clean};
  for (const void* q : all)
    if (q && !aligned16(q)) return CSBP_ERR_INVALID;
  const WsLayout wl = ws_layout(problem, 1);
  if (ws_bytes < wl.total) return CSBP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const csbp_problem& p = *problem;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dsum = reinterpret_cast<float*>(ws + wl.dsum);
  float* dq_acc = reinterpret_cast<float*>(ws + wl.dq_acc);

  CUtensorMap maps[11];
  const int qi = in->q_clean ? 0 : 3;  // the clean-query maps are unused when absent
  const void* qc = in->q_clean ? in->q_clean : in->q_corr;
  const void* dc = do_clean ? do_clean : do_corr;
  const TokStride dos = contiguous_stride(p.Hq, p.d, p.L);
  const int qbox = bwd_query_box_rows();
  if (!make_map_dqacc(&maps[10], dq_acc, p.Hq, p.d, p.L, 2 * static_cast<int64_t>(p.batch),
                      bwd_dq_box_rows(p.d)))
    return CSBP_ERR_CUDA;
  if (!make_map(&maps[0], qc, p.Hq, p.d, p.L, p.batch, input_stride(problem, in, qi), qbox) ||
      !make_map(&maps[1], in->q_corr, p.Hq, p.d, p.L, p.batch, input_stride(problem, in, 3),
                qbox) ||
      !make_map(&maps[2], in->k_clean, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 1)) ||
      !make_map(&maps[3], in->k_corr, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 4)) ||
      !make_map(&maps[4], in->v_clean, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 2)) ||
      !make_map(&maps[5], in->v_corr, p.Hkv, p.d, p.L, p.batch, input_stride(problem, in, 5)) ||
      !make_map(&maps[6], dc, p.Hq, p.d, p.L, p.batch, dos, qbox) ||
      !make_map(&maps[7], do_corr, p.Hq, p.d, p.L, p.batch, dos, qbox) ||
      !make_map_rows_f32(&maps[8], lse, p.L, static_cast<int64_t>(p.batch) * 2 * p.Hq, qbox) ||
      !make_map_rows_f32(&maps[9], dsum, p.L, static_cast<int64_t>(p.batch) * 2 * p.Hq, qbox))
    return CSBP_ERR_CUDA;
  const int64_t rows = static_cast<int64_t>(p.batch) * p.L;
  const int64_t stream_elems = rows * p.Hq * p.d;
  const void* o_s[2] = {o_clean, o_corr};
  const void* do_s[2] = {do_clean, do_corr};
  for (int qs = hc ? 0 : 1; qs < 2; ++qs) {
    const int tp = timer_begin(7, stream);
    const cudaError_t pe = launch_bwd_pre(p.d, o_s[qs], do_s[qs], dsum + qs * rows * p.Hq,
                                          dq_acc + qs * stream_elems, rows, p.Hq, p.L, stream);
    timer_end(tp, stream);
    if (pe != cudaSuccess)
      return CSBP_ERR_CUDA;
  }

  const WorkOffsets wo = work_offsets(info);
  BwdParams bp;
  bp.tasks = static_cast<const int32_t*>(work_dev) + wo.bwd_tasks;
  bp.segs = static_cast<const int32_t*>(work_dev) + wo.bwd_segs;
  bp.L = p.L;
  bp.M = p.M;
  bp.Hq = p.Hq;
  bp.Hkv = p.Hkv;
  bp.G = p.Hq / p.Hkv;
  bp.batch = p.batch;
  bp.window = p.window;
  bp.clean_causal = p.clean_causal;
  bp.n_segs = info->n_bwd_segments;
  bp.nT = (p.L + kTile - 1) / kTile;
  bp.scale_log2 = p.scale * 1.4426950408889634f;
  bp.scale = p.scale;
  bp.dq_acc = dq_acc;
  bp.dk[0] = dk_clean;
  bp.dk[1] = dk_corr;
  bp.dv[0] = dv_clean;
  bp.dv[1] = dv_corr;
  bp.status = reinterpret_cast<int*>(ws + wl.status);
  bp.dk_acc = nullptr;
  bp.dv_acc = nullptr;
  const bool windowed = bwd_windowed(problem);
  const int64_t kv_elems = rows * p.Hkv * p.d;  // per key stream
  if (windowed) {
    bp.dk_acc = reinterpret_cast<float*>(ws + wl.dk_acc);
    bp.dv_acc = reinterpret_cast<float*>(ws + wl.dv_acc);
    if (launch_fill(bp.dk_acc, 2 * kv_elems, 0.f, stream) != cudaSuccess ||
        launch_fill(bp.dv_acc, 2 * kv_elems, 0.f, stream) != cudaSuccess)
      return CSBP_ERR_CUDA;
  }
  // KV-head-major CTA order once each KV head has at least four waves of
  // tasks (measured: +33 % on a 128K corrupted-only backward, -8 % on a 16K
  // two-copy one, where a KV head's tasks span less than two waves)
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CSBP_ERR_CUDA;
    bp.kv_major = (static_cast<int64_t>(info->n_bwd_tasks) >= 4 * static_cast<int64_t>(sms)) ? 1 : 0;
  }
  const int timed = timer_begin(1, stream);
  const cudaError_t be = launch_bwd(p.d, maps, bp, info->n_bwd_tasks, stream);
  timer_end(timed, stream);
  if (be != cudaSuccess) return CSBP_ERR_CUDA;

  if (windowed) {
    void* dk_s[2] = {dk_clean, dk_corr};
    void* dv_s[2] = {dv_clean, dv_corr};
    for (int ks = 0; ks < 2; ++ks) {
      const int tc = timer_begin(9, stream);
      const cudaError_t ce =
          launch_dq_convert(bp.dk_acc + ks * kv_elems, dk_s[ks], kv_elems, 1.f, stream) != cudaSuccess
              ? cudaErrorUnknown
              : launch_dq_convert(bp.dv_acc + ks * kv_elems, dv_s[ks], kv_elems, 1.f, stream);
      timer_end(tc, stream);
      if (ce != cudaSuccess) return CSBP_ERR_CUDA;
    }
  }
  void* dq_s[2] = {dq_clean, dq_corr};
  for (int qs = hc ? 0 : 1; qs < 2; ++qs) {
    const int tq = timer_begin(8, stream);
    const cudaError_t qe = launch_dq_convert(dq_acc + qs * stream_elems, dq_s[qs], stream_elems,
                                             p.scale, stream);
    timer_end(tq, stream);
    if (qe != cudaSuccess) return CSBP_ERR_CUDA;
  }
  return CSBP_OK;
}

extern "C" csbp_status csbp_lse_merge(int32_t n_parts, const float* const* o_parts,
                                      const float* const* lse_parts, int64_t rows, int32_t Hq,
                                      int32_t d, void* o_out, float* lse_out, void* stream) {
  if (n_parts < 1 || n_parts > kMaxParts || rows < 1 || Hq < 1 || d < 4 || d % 4 != 0)
    return CSBP_ERR_INVALID;
  // rows x Hq x d below 2^39 elements, tested by division (no overflow)
  constexpr int64_t kMaxElems = int64_t(1) << 39;
  if (rows > (kMaxElems - 1) / Hq || rows * Hq > (kMaxElems - 1) / d) return CSBP_ERR_INVALID;
  if (!o_parts || !lse_parts || !o_out || !lse_out) return CSBP_ERR_INVALID;
  if (!aligned16(o_out) && (d % 8 != 0 || (reinterpret_cast<uintptr_t>(o_out) & 7u)))
    return CSBP_ERR_INVALID;
  const auto aligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  if (!aligned4(lse_out)) return CSBP_ERR_INVALID;  // fp32 LSE rows
  MergeArgs a;
  for (int s = 0; s < n_parts; ++s) {
    if (!o_parts[s] || !lse_parts[s] || !aligned16(o_parts[s]) || !aligned4(lse_parts[s]))
      return CSBP_ERR_INVALID;
    a.o[s] = o_parts[s];
    a.z[s] = lse_parts[s];
  }
  if (launch_lse_merge(a, n_parts, rows, Hq, d, o_out, lse_out,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CSBP_ERR_CUDA;
  return CSBP_OK;
}

extern "C" csbp_status csbp_e4m3_to_bf16(const void* in, float scale, void* out, int64_t n,
                                         void* stream) {
  constexpr int64_t kMaxElems = int64_t(1) << 40;
  if (!in || !out || n < 0 || n >= kMaxElems) return CSBP_ERR_INVALID;
  if (!(scale == scale) || scale == 0.f || scale > 3.0e38f || scale < -3.0e38f)
    return CSBP_ERR_INVALID;  // NaN, zero or infinite
  if (!aligned16(in) || !aligned16(out)) return CSBP_ERR_INVALID;
  if (n == 0) return CSBP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int tk = timer_begin(10, s);
  const cudaError_t e = launch_e4m3_to_bf16(in, out, n, scale, s);
  timer_end(tk, s);
  return e == cudaSuccess ? CSBP_OK : CSBP_ERR_CUDA;
}

extern "C" csbp_status csbp_check_status(void* workspace, void* stream) {
  if (!workspace) return CSBP_ERR_INVALID;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSBP_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CSBP_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return CSBP_ERR_CUDA;
    // device codes: 1 timeout, 2 misaligned window, 3 bad work record (debug builds)
    return v == 1 ? CSBP_ERR_TIMEOUT : CSBP_ERR_DEVICE;
  }
  return CSBP_OK;
}
