// Fused two-copy block-diffusion attention, forward, for sm_103a.
//
// Computes, per query row of either copy, softmax(scale * q K^T + mask) V over
// exactly the keys the block-diffusion mask allows ("CSBP 完全拆解" blog,
// section "CSBP：BP 管损坏块，CP 管干净上下文": O_b = Attn(Q_b, [K_b; K^clean_<b],
// [V_b; V^clean_<b]); clean queries block-causal over the clean copy), and the
// row's natural-log softmax denominator (LSE).  Partial mode writes one
// normalised fp32 partial per key part for the exact LSE merge of the
// section "在线 softmax 合并：为什么分两段算仍是同一个注意力".
//
// One CTA owns two consecutive work-list tasks of one (batch, query head):
// two 128-row query tiles ("slots").  The list is sorted heaviest first, and
// equal-cost tasks of one key part and query copy are adjacent, so the two
// usually read the same key tiles.  It walks the union of their key tiles in (copy,
// tile) order, so a key tile both slots read is loaded once.  Each slot has
// its own softmax warpgroup, and the two keep the tensor pipe busy in turn:
// while one slot's softmax runs, the other slot's MMAs do.  Roles (384
// threads):
//   warp 0 lane 0  TMA producer: both Q tiles once, then K / V of each key
//                  tile of the union into 2-stage rings
//   warp 1 lane 0  MMA issuer (it polls the two waits on its chain: a PV's
//                  completion before the S that overwrites its P, and the
//                  softmax's P before its PV), per key tile of the union and
//                  slot by slot:
//                  O_s += P_s V of the previous tile, then S_s = Q_s K^T of
//                  this one (once that PV has read the P_s it overwrites)
//   warps 4..7, 8..11  softmax of slot 0, 1: thread t owns query row t (TMEM
//                  lane t); reads S with tcgen05.ld, masks partial tiles,
//                  keeps a running reference max, writes P (bf16 pairs) back
//                  over the first 64 columns of its S, which the PV MMA reads
//                  as its A operand, and rescales the TMEM accumulator only
//                  when the row max grows by more than 2^8 (exact: O and l
//                  share the reference).
// TMEM columns: S of slot s at 128 s, O of slot s at 256 + d s.  All shared
// state lives in the dynamic window, which must start 1024-byte aligned.
#include <cuda.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"
#include "device_once.h"
#include "mbar_spin.cuh"
#include "pair_math.cuh"
#include "ptx_sm100.cuh"
#include "work_checks.cuh"

namespace csbp {

namespace {

constexpr int kThreads = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Per-warpgroup register budgets (setmaxnreg): producer / MMA, softmax.
// Their sum must not exceed the launch allocation (checked on the host).
constexpr uint32_t kRegsLow = 112;
constexpr uint32_t kRegsSoftmax = 192;
constexpr int kRegsNeeded = 128 * kRegsLow + 256 * kRegsSoftmax;

enum FwdBar {
  B_Q_FULL = 0,               // [2] per slot
  B_K_FULL = B_Q_FULL + 2,    // [2] ring stage
  B_K_EMPTY = B_K_FULL + 2,   // [2]
  B_V_FULL = B_K_EMPTY + 2,   // [2]
  B_V_EMPTY = B_V_FULL + 2,   // [2]
  B_S_FULL = B_V_EMPTY + 2,   // [2] per slot
  B_P_FULL = B_S_FULL + 2,    // [2] per slot (its four softmax warps)
  B_PV_DONE = B_P_FULL + 2,   // [2] per slot
  B_DRAIN = B_PV_DONE + 2,
  B_COUNT
};

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;     // Q/K/V tile (bf16)
  static constexpr int kBoxBytes = kTile * 64 * 2;     // one 64-column TMA box
  static constexpr int kQ = 0;                         // 2 slots
  static constexpr int kK = kQ + 2 * kTileBytes;       // 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;       // 2 stages
  static constexpr int kBar = kV + 2 * kTileBytes;
  static constexpr int kMisc = kBar + B_COUNT * 8;     // tmem base, abort flag
  static constexpr int kDynSmem = kMisc + 16;
  static constexpr uint32_t kColO = 256;               // O of slot s at kColO + D s
};

// Walk over the key tiles of one task's segments, in (copy, tile) order.
struct SlotWalk {
  const int32_t* seg;
  int segs_left, left;  // segments after the current one, tiles not yet passed
  int stream, t, end, flags;
  __device__ void start(const int32_t* s, int n_segs, int n_tiles) {
    seg = s;
    segs_left = n_segs;
    left = n_tiles;
    stream = t = end = flags = 0;
    load();
  }
  __device__ void load() {
    if (segs_left <= 0) return;
    stream = seg[0];
    t = seg[1];
    end = seg[2];
    flags = seg[3];
    seg += kSegWords;
    --segs_left;
  }
  __device__ int key() const { return left > 0 ? (stream << 24) + t : 0x7fffffff; }
  __device__ void next() {
    --left;
    if (++t >= end) load();
  }
};

// Walk over the union of two slots' key tiles: which slots read the current
// tile, and its copy and index.
struct PairWalk {
  SlotWalk w[2];
  int in0, in1, stream, t;
  __device__ void settle() {
    const int k0 = w[0].key(), k1 = w[1].key();
    const int k = min(k0, k1);
    in0 = (k0 == k) && k != 0x7fffffff;
    in1 = (k1 == k) && k != 0x7fffffff;
    stream = in0 ? w[0].stream : w[1].stream;
    t = in0 ? w[0].t : w[1].t;
  }
  __device__ bool valid() const { return in0 || in1; }
  __device__ void next() {
    if (in0) w[0].next();
    if (in1) w[1].next();
    settle();
  }
};

// Key positions [lo, hi) of copy k_stream that query position qpos (block qb)
// of copy q_stream may read: clean queries read clean keys of blocks <= qb
// (keys <= qpos when token-causal); corrupted queries read clean keys of
// blocks < qb and the corrupted keys of their own block; a window W > 0 also
// drops keys W or more positions back.
__device__ __forceinline__ void allowed_key_range(int q_stream, int k_stream, int qpos, int qb,
                                                  int M, int L, int window, int clean_causal,
                                                  bool row_valid, int& lo, int& hi) {
  lo = 0;
  if (!row_valid || (q_stream == 0 && k_stream == 1)) {
    hi = 0;
    return;
  }
  if (q_stream == 0) {
    hi = clean_causal ? qpos + 1 : (qb + 1) * M;
  } else if (k_stream == 0) {
    hi = qb * M;
  } else {
    lo = qb * M;
    hi = (qb + 1) * M;
  }
  hi = min(hi, L);
  if (window > 0) lo = max(lo, qpos - window + 1);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
               const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
               const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
               const FwdParams p, int n_tasks) {
  using Lay = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // layout below needs a 1024-aligned window
    if (threadIdx.x == 0) atomicExch(p.status, DEV_MISALIGNED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Lay::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- decode the unit: (task pair, batch, query head)
  const int hb = p.Hq * p.batch;
  const int pair = blockIdx.x / hb;
  const int rem = blockIdx.x - pair * hb;
  const int bz = rem / p.Hq;
  const int h = rem - bz * p.Hq;
  const int kvh = h / p.G;
  const int n_slots = (2 * pair + 1 < n_tasks) ? 2 : 1;
  auto task_words = [&](int s) { return p.tasks + static_cast<int64_t>(2 * pair + s) * kTaskWords; };
  auto slot_walk = [&](int s, SlotWalk& w) {
    if (s < n_slots) {
      const int32_t* tw = task_words(s);
      w.start(p.segs + static_cast<int64_t>(tw[3]) * kSegWords, tw[4], tw[5]);
    } else {
      w.start(nullptr, 0, 0);
    }
  };
  auto slot_tiles = [&](int s) { return s < n_slots ? task_words(s)[5] : 0; };
#ifdef CSBP_DEBUG_CHECKS
  {
    bool bad = false;
    if (threadIdx.x == 0) {
      for (int s = 0; s < n_slots; ++s)
        if (!task_record_ok(task_words(s), p.segs, p.n_segs, p.nT)) bad = true;
      if (bad) atomicExch(p.status, DEV_BADWORK);
    }
    if (__syncthreads_or(bad)) return;  // nothing issued yet
  }
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i)
      mbar_init(&bars[i], (i >= B_P_FULL && i < B_P_FULL + 2) ? 4 : 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_sh;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ===================== TMA producer
      prefetch_tmap(&tm_q0);
      prefetch_tmap(&tm_q1);
      prefetch_tmap(&tm_k0);
      prefetch_tmap(&tm_k1);
      prefetch_tmap(&tm_v0);
      prefetch_tmap(&tm_v1);
      for (int s = 0; s < n_slots; ++s) {
        const int32_t* tw = task_words(s);
        const void* tq = tw[0] ? static_cast<const void*>(&tm_q1) : static_cast<const void*>(&tm_q0);
        mbar_arrive_expect_tx(&bars[B_Q_FULL + s], Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kQ + s * Lay::kTileBytes + c * Lay::kBoxBytes, tq,
                      &bars[B_Q_FULL + s], h * D + c * 64, tw[1] * kTile, bz);
      }
      PairWalk w;
      slot_walk(0, w.w[0]);
      slot_walk(1, w.w[1]);
      w.settle();
      int nk = 0, nv = 0;  // K / V tiles whose loads were issued
      bool ok = true;
      for (int m = 0; w.valid() && ok; ++m, w.next()) {
        const int b = m & 1;
        const void* tk = w.stream ? static_cast<const void*>(&tm_k1) : static_cast<const void*>(&tm_k0);
        const void* tv = w.stream ? static_cast<const void*>(&tm_v1) : static_cast<const void*>(&tm_v0);
        if (m >= 2) ok = mbar_wait(&bars[B_K_EMPTY + b], ((m - 2) >> 1) & 1, p.status, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[B_K_FULL + b], Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kK + b * Lay::kTileBytes + c * Lay::kBoxBytes, tk,
                      &bars[B_K_FULL + b], kvh * D + c * 64, w.t * kTile, bz);
        nk = m + 1;
        if (m >= 2) ok = mbar_wait(&bars[B_V_EMPTY + b], ((m - 2) >> 1) & 1, p.status, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[B_V_FULL + b], Lay::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + Lay::kV + b * Lay::kTileBytes + c * Lay::kBoxBytes, tv,
                      &bars[B_V_FULL + b], kvh * D + c * 64, w.t * kTile, bz);
        nv = m + 1;
      }
      if (!ok) {
        // drain: wait (ignoring the abort flag) for the loads already issued
        for (int s = 0; s < n_slots; ++s)
          mbar_wait(&bars[B_Q_FULL + s], 0, nullptr, nullptr, 200000000ull);
        for (int m = (nk > 2 ? nk - 2 : 0); m < nk; ++m)
          mbar_wait(&bars[B_K_FULL + (m & 1)], (m >> 1) & 1, nullptr, nullptr, 200000000ull);
        for (int m = (nv > 2 ? nv - 2 : 0); m < nv; ++m)
          mbar_wait(&bars[B_V_FULL + (m & 1)], (m >> 1) & 1, nullptr, nullptr, 200000000ull);
      }
    } else if (warp == 1 && lane == 0) {
      // ===================== MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      bool ok = true;
      for (int s = 0; s < n_slots && ok; ++s) ok = mbar_wait(&bars[B_Q_FULL + s], 0, p.status, abort_flag);
      int npv[2] = {0, 0};  // PV issued per slot
      // S_s = Q_s K^T of ring stage b into slot s's S columns
      auto issue_s = [&](int s, int b) -> bool {
        if (npv[s] > 0 &&
            !mbar_wait_spin(&bars[B_PV_DONE + s], (npv[s] - 1) & 1, p.status, abort_flag))
          return false;  // its last PV still reads the P held there
        tc_fence_after_sync();
        const uint64_t q_desc = sdesc_sw128(smem_u32(smem + Lay::kQ + s * Lay::kTileBytes), 16, 1024);
        const uint64_t k_desc = sdesc_sw128(smem_u32(smem + Lay::kK + b * Lay::kTileBytes), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * Lay::kBoxBytes + (k & 3) * 32;
          umma_bf16_ss(tmem + s * 128, sdesc_step(q_desc, off), sdesc_step(k_desc, off), idesc_s,
                       k > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_S_FULL + s]);
        return true;
      };
      // O_s += P_s V of ring stage b, P_s (bf16 pairs) in slot s's S columns
      auto issue_pv = [&](int s, int b) -> bool {
        if (!mbar_wait_spin(&bars[B_P_FULL + s], npv[s] & 1, p.status, abort_flag)) return false;
        tc_fence_after_sync();
        const uint64_t vb = sdesc_sw128(smem_u32(smem + Lay::kV + b * Lay::kTileBytes), Lay::kBoxBytes,
                                        1024);  // V, MN-major B
        const uint32_t acc0 = npv[s] > 0 ? 1u : 0u;
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
          umma_bf16_ts(tmem + Lay::kColO + s * D, tmem + s * 128 + k * 8, sdesc_step(vb, k * 2048),
                       idesc_pv, k > 0 ? 1u : acc0);
        umma_commit(&bars[B_PV_DONE + s]);
        ++npv[s];
        return true;
      };
      PairWalk w;
      slot_walk(0, w.w[0]);
      slot_walk(1, w.w[1]);
      w.settle();
      int prev_in[2] = {0, 0};
      int m = 0;
      // Per key tile m: PV_0 of tile m-1, S_0 of tile m, PV_1 of tile m-1,
      // S_1 of tile m.  Every S_s waits for the PV_s before it (P_s shares
      // its columns), and that wait idles the tensor pipe; the other waits
      // of the tile (K_m, the walk to the next tile) sit inside those two
      // drains instead of between MMA groups.
      for (; w.valid() && ok; ++m) {
        const int b = m & 1;
        const int pb = (m - 1) & 1;
        const int in[2] = {w.in0, w.in1};
        if (m > 0) ok = mbar_wait(&bars[B_V_FULL + pb], ((m - 1) >> 1) & 1, p.status, abort_flag);
        if (ok && prev_in[0]) ok = issue_pv(0, pb);
        if (ok) ok = mbar_wait(&bars[B_K_FULL + b], (m >> 1) & 1, p.status, abort_flag);
        if (ok && in[0]) ok = issue_s(0, b);
        if (ok && prev_in[1]) ok = issue_pv(1, pb);
        if (!ok) break;
        if (m > 0) umma_commit(&bars[B_V_EMPTY + pb]);
        w.next();
        if (in[1]) ok = issue_s(1, b);
        if (!ok) break;
        umma_commit(&bars[B_K_EMPTY + b]);
        prev_in[0] = in[0];
        prev_in[1] = in[1];
      }
      if (ok && m > 0) {
        const int pb = (m - 1) & 1;
        ok = mbar_wait(&bars[B_V_FULL + pb], ((m - 1) >> 1) & 1, p.status, abort_flag);
        for (int s = 0; s < 2 && ok; ++s)
          if (prev_in[s]) ok = issue_pv(s, pb);
      }
      // drain every MMA this thread issued before the CTA may free TMEM
      umma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, nullptr, nullptr, 500000000ull);
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ===================== softmax warpgroup of slot s
    const int s = (warp - 4) >> 2;
    const int row = threadIdx.x - 128 * (1 + s);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t colS = s * 128;
    const uint32_t colO = Lay::kColO + s * D;
    const int n_tiles = slot_tiles(s);
    if (n_tiles > 0) {
      const int32_t* tw = task_words(s);
      const int q_stream = tw[0];
      const int q_tile = tw[1];
      const int part = tw[2];
      const int64_t qpos = static_cast<int64_t>(q_tile) * kTile + row;
      const bool row_valid = qpos < p.L;
      const int qb = row_valid ? static_cast<int>(qpos) / p.M : -1;
      const float sl2 = p.scale_log2;
      float m_ref = -INFINITY;
      float l = 0.f;
      SlotWalk w;
      slot_walk(s, w);
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j, w.next()) {
        if (!mbar_wait_warp(&bars[B_S_FULL + s], j & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        float sv[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; c += 2)
          tmem_ld32x2(tmem + lane_base + colS + c * 32, tmem + lane_base + colS + (c + 1) * 32,
                      sv + c * 32, sv + (c + 1) * 32);
        const bool ragged = (static_cast<int64_t>(w.t) + 1) * kTile > p.L;
        float mx = -INFINITY;
        // bit q: no row of this warp may read a key of 32-column chunk q
        // (warp-uniform): the max skips it, and a 64-column half with both
        // chunks dead gets P = 0 without its exponentials
        uint32_t dead = 0;
        // warp-uniform: the votes below need every lane of the warp (rows
        // past L make row_valid differ inside the last query tile)
        if (__any_sync(0xffffffffu, (w.flags & 1) || ragged || !row_valid)) {
          // the allowed keys of this query row form one range [lo, hi)
          int lo, hi;
          allowed_key_range(q_stream, w.stream, static_cast<int>(qpos), qb, p.M, p.L, p.window,
                            p.clean_causal, row_valid, lo, hi);
          lo -= w.t * kTile;
          hi -= w.t * kTile;
#pragma unroll
          for (int q = 0; q < kTile / 32; ++q) {
            const int c0 = q * 32;
            if (__all_sync(0xffffffffu, hi <= c0 || lo >= c0 + 32)) {
              dead |= 1u << q;
#pragma unroll
              for (int c = c0; c < c0 + 32; ++c) sv[c] = -INFINITY;
            } else if (!__all_sync(0xffffffffu, lo <= c0 && hi >= c0 + 32)) {
#pragma unroll
              for (int c = c0; c < c0 + 32; ++c) sv[c] = (c >= lo && c < hi) ? sv[c] : -INFINITY;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kTile / 32; ++q) {
          if (dead & (1u << q)) continue;
#pragma unroll
          for (int c = q * 32; c < q * 32 + 32; c += 2) mx = fmax3(mx, sv[c], sv[c + 1]);
        }
        // scores stay unscaled: the scale is positive, so the row max of the
        // scaled scores is the scaled max, and each exponent below takes the
        // scale in one fused multiply-add
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool need = m_new > m_ref + kRescaleThreshold;  // false while both are -inf
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O holds PV_0..PV_{j-1} scaled by the old reference; PV_{j-1} is
          // complete: the S this tile read was issued after it
          const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_base + colO + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + lane_base + colO + c * 32, o);
          }
        }
        if (need) {
          l *= exp2f(m_ref - m_new);  // 0 when m_ref was -inf
          m_ref = m_new;
        }
        const float mref_safe = (m_ref == -INFINITY) ? 0.f : m_ref;
        // exponent arguments and the row sum two lanes per instruction
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm = f2_pack(-mref_safe, -mref_safe);
        uint64_t rs2 = f2_pack(0.f, 0.f);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float packed[32];
          if (((dead >> (2 * half)) & 3u) == 3u) {
#pragma unroll
            for (int c = 0; c < 32; ++c) packed[c] = 0.f;
            tmem_st32(tmem + lane_base + colS + half * 32, packed);
            continue;
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[half * 64 + 2 * c], sv[half * 64 + 2 * c + 1]), sl2x2, negm),
                      x0, x1);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            rs2 = f2_add(rs2, f2_pack(e0, e1));
            packed[c] = __uint_as_float(pack_bf16x2(e0, e1));
          }
          tmem_st32(tmem + lane_base + colS + half * 32, packed);
        }
        float rs0, rs1;
        f2_unpack(rs2, rs0, rs1);
        l += rs0 + rs1;
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_P_FULL + s]);
      }
      // ---- epilogue: wait for the last PV, normalise, store
      if (ok && mbar_wait_warp(&bars[B_PV_DONE + s], (n_tiles - 1) & 1, p.status, abort_flag)) {
        tc_fence_after_sync();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        const float lse = (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (p.partial_mode) {
          const int64_t prow = ((static_cast<int64_t>(part) * 2 + q_stream) * p.batch + bz);
          float* dst = p.part_o + (prow * p.L + qpos) * p.Hq * D + static_cast<int64_t>(h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_base + colO + c * 32, o);
            if (row_valid) {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + c * 32 + i) =
                    make_float4(o[i] * inv_l, o[i + 1] * inv_l, o[i + 2] * inv_l, o[i + 3] * inv_l);
            }
          }
          if (row_valid) p.part_lse[(prow * p.Hq + h) * p.L + qpos] = lse;
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(q_stream ? p.o[1] : p.o[0]) +
                               ((static_cast<int64_t>(bz) * p.L + qpos) * p.Hq + h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_base + colO + c * 32, o);
            if (row_valid) {
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 v;
                v.x = pack_bf16x2(o[i] * inv_l, o[i + 1] * inv_l);
                v.y = pack_bf16x2(o[i + 2] * inv_l, o[i + 3] * inv_l);
                v.z = pack_bf16x2(o[i + 4] * inv_l, o[i + 5] * inv_l);
                v.w = pack_bf16x2(o[i + 6] * inv_l, o[i + 7] * inv_l);
                *reinterpret_cast<uint4*>(dst + c * 32 + i) = v;
              }
            }
          }
          if (row_valid)
            p.lse[((static_cast<int64_t>(bz) * 2 + q_stream) * p.Hq + h) * p.L + qpos] = lse;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap* maps, const FwdParams& p, int n_tasks,
                                cudaStream_t stream) {
  using Lay = FwdLayout<D>;
  // the shared-memory limit is a per-device attribute: set it once on each
  // device, and read the kernel's register count there
  static PerDeviceOnce configured;
  static int launch_regs[PerDeviceOnce::kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!configured.run(dev, [&](int device) {
        e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Lay::kDynSmem);
        if (e != cudaSuccess) return false;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, fwd_kernel<D>);
        if (e != cudaSuccess) return false;
        launch_regs[device] = fa.numRegs;
        return true;
      }))
    return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  // setmaxnreg.inc would wait forever if the budgets exceeded the launch
  // allocation: refuse to launch instead
  if (launch_regs[dev] * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  const int64_t grid = static_cast<int64_t>((n_tasks + 1) / 2) * p.Hq * p.batch;
  if (grid <= 0) return cudaSuccess;
  fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, Lay::kDynSmem, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p, n_tasks);
  return cudaGetLastError();
}

// maps: q_clean, q_corr, k_clean, k_corr, v_clean, v_corr
cudaError_t launch_fwd(int d, const CUtensorMap* maps, const FwdParams& p, int n_tasks,
                       cudaStream_t stream) {
  if (d == 128) return launch_fwd_d<128>(maps, p, n_tasks, stream);
  return launch_fwd_d<64>(maps, p, n_tasks, stream);
}

}  // namespace csbp
