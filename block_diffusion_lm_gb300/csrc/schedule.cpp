// Host-side ownership and mask-aware tile scheduling (csbp_block_schedule).
//
// Ownership follows the dual-end pairing of the "CSBP 完全拆解" blog, section
// "负载均衡：为什么要首尾块配对", and the Turbo-dLLM project page, section "Load
// balancing: pairing early and late blocks": the clean sequence is cut into
// 2P contiguous chunks, shard r owns chunks r and 2P-1-r, and a corrupted
// block belongs to the owner of the clean chunk holding its first position.
//
// The tile work list enumerates only the (query tile, key tile) pairs that
// hold at least one entry allowed by the block-diffusion mask ("传统上下文并行
// 为什么会传错东西" section of the same blog: a corrupted query of block b reads
// its own block's corrupted keys and the clean keys of blocks < b; clean
// queries read clean keys of blocks <= b).  Classification of a tile pair is
// analytic on block-id intervals, and each tile's candidates are the span
// between its first and last position's allowed ranges, so building the list
// costs about one classification per listed pair, with no mask materialised.
#include <algorithm>
#include <cstring>
#include <vector>

#include "csbp.h"
#include "csbp_internal.h"

namespace csbp {

// Allowed key positions [lo, hi) of copy k_stream for query position i of
// copy q_stream, with the optional window (keys less than `window` positions
// back) and token-causal clean attention; both bounds are non-decreasing in i.
void key_range(int q_stream, int k_stream, int64_t i, int64_t L, int64_t M, int64_t window,
               bool clean_causal, int64_t& lo, int64_t& hi) {
  const int64_t b = i / M;
  lo = 0;
  if (q_stream == 0 && k_stream == 1) {
    hi = 0;
    return;
  }
  if (q_stream == 0) {
    hi = clean_causal ? i + 1 : std::min((b + 1) * M, L);
  } else if (k_stream == 0) {
    hi = b * M;
  } else {
    lo = b * M;
    hi = std::min((b + 1) * M, L);
  }
  if (window > 0) lo = std::max(lo, i - window + 1);
}

// Allowed query positions [lo, hi) of copy q_stream that may read key
// position j of copy k_stream (the transpose of key_range); both bounds are
// non-decreasing in j.
void query_range(int q_stream, int k_stream, int64_t j, int64_t L, int64_t M, int64_t window,
                 bool clean_causal, int64_t& lo, int64_t& hi) {
  const int64_t b = j / M;
  hi = L;
  if (q_stream == 0 && k_stream == 1) {
    lo = hi = 0;
    return;
  }
  if (k_stream == 0) {
    lo = (q_stream == 0) ? (clean_causal ? j : b * M) : (b + 1) * M;
  } else {
    lo = b * M;
    hi = std::min((b + 1) * M, L);
  }
  if (window > 0) hi = std::min(hi, j + window);
}

// Tiles of the other copy that can hold an allowed entry for tile t: the
// first position's lower bound to the last position's upper bound (both
// bounds are non-decreasing, so every position's range lies inside), as a
// half-open tile range [a, b).
template <typename RangeFn>
void tile_span(RangeFn range, int64_t t, int64_t L, int64_t T, int64_t& a, int64_t& b) {
  const int64_t p0 = t * T, p1 = std::min(p0 + T, L) - 1;
  int64_t lo0, hi0, lo1, hi1;
  range(p0, lo0, hi0);
  range(p1, lo1, hi1);
  if (p0 > p1 || hi1 <= lo0) {
    a = b = 0;
    return;
  }
  a = lo0 / T;
  b = (hi1 - 1) / T + 1;
}

// 0 = no allowed entry, 1 = some (partial), 2 = all entries allowed; from the
// rows' key ranges (non-decreasing, so the first and last rows bound the
// hull and the tightest row; only tiles between the two are scanned)
int classify_tile_ranges(int q_stream, int64_t qt, int k_stream, int64_t kt, int64_t L,
                         int64_t M, int64_t T, int64_t window, bool clean_causal) {
  const int64_t r0 = qt * T, r1 = std::min(r0 + T, L) - 1;
  const int64_t c0 = kt * T, c1 = std::min(c0 + T, L) - 1;
  if (r0 > r1 || c0 > c1) return 0;
  int64_t lo0, hi0, lo1, hi1;
  key_range(q_stream, k_stream, r0, L, M, window, clean_causal, lo0, hi0);
  key_range(q_stream, k_stream, r1, L, M, window, clean_causal, lo1, hi1);
  if (lo0 > c1 || hi1 <= c0) return 0;      // outside every row's range
  if (lo1 <= c0 && hi0 > c1) return 2;      // inside every row's range
  for (int64_t i = r0; i <= r1; ++i) {
    int64_t lo, hi;
    key_range(q_stream, k_stream, i, L, M, window, clean_causal, lo, hi);
    if (lo <= c1 && hi > c0 && lo < hi) return 1;
  }
  return 0;
}

// 0 = no allowed entry, 1 = some (partial), 2 = all entries allowed.
int classify_tile(int q_stream, int64_t qt, int k_stream, int64_t kt, int64_t L, int64_t M,
                  int64_t T) {
  const int64_t r0 = qt * T, r1 = std::min(r0 + T, L) - 1;
  const int64_t c0 = kt * T, c1 = std::min(c0 + T, L) - 1;
  if (r0 > r1 || c0 > c1) return 0;
  const int64_t bq0 = r0 / M, bq1 = r1 / M, bk0 = c0 / M, bk1 = c1 / M;
  if (q_stream == 0 && k_stream == 1) return 0;  // clean q never reads corrupted k
  if (q_stream == 0) {                           // clean-clean: bk <= bq
    if (bk0 > bq1) return 0;
    return bk1 <= bq0 ? 2 : 1;
  }
  if (k_stream == 0) {  // corrupted q, clean k: bk < bq
    if (bk0 >= bq1) return 0;
    return bk1 < bq0 ? 2 : 1;
  }
  // corrupted q, corrupted k: bk == bq
  if (bk1 < bq0 || bk0 > bq1) return 0;
  return (bk0 == bk1 && bq0 == bq1 && bk0 == bq0) ? 2 : 1;
}

namespace {

struct Seg {
  int32_t stream, begin, end, flags;
};
struct Task {
  int32_t a_stream, a_tile, part;
  std::vector<Seg> segs;
  int32_t cost;
  int64_t canon;
  int32_t flags = 0;   // bwd: bit0 = dK/dV into the fp32 accumulators
  int32_t window = 0;  // bwd: query-tile window, 0 = the last one
};

// Append tile `t` with class `cls` (1/2) of `stream` to a run-length list of
// homogeneous segments (same stream, same partial flag, same part).
void push_tile(std::vector<Seg>& segs, std::vector<int32_t>& seg_part, int32_t stream,
               int32_t t, int cls, int32_t part) {
  const int32_t flags = (cls == 1) ? 1 : 0;
  if (!segs.empty()) {
    Seg& s = segs.back();
    if (s.stream == stream && s.end == t && s.flags == flags && seg_part.back() == part) {
      s.end = t + 1;
      return;
    }
  }
  segs.push_back({stream, t, t + 1, flags});
  seg_part.push_back(part);
}

}  // namespace

csbp_status validate_problem(const csbp_problem* p) {
  if (!p) return CSBP_ERR_INVALID;
  if (p->batch < 1 || p->L < 1 || p->M < 1 || p->Hq < 1 || p->Hkv < 1 || p->P < 1)
    return CSBP_ERR_INVALID;
  if (p->L % p->M != 0) return CSBP_ERR_INVALID;
  if (p->Hq % p->Hkv != 0) return CSBP_ERR_INVALID;
  if (!(p->scale > 0.0f) || p->scale != p->scale) return CSBP_ERR_INVALID;
  if (p->tile_q < 1 || p->tile_kv < 1) return CSBP_ERR_INVALID;
  if (p->has_clean_queries != 0 && p->has_clean_queries != 1) return CSBP_ERR_INVALID;
  if (p->window < 0 || (p->clean_causal != 0 && p->clean_causal != 1)) return CSBP_ERR_INVALID;
  if (p->bwd_chunk < 0) return CSBP_ERR_INVALID;
  if (p->per_rank != 0 && p->per_rank != 1) return CSBP_ERR_INVALID;
  if (p->per_rank ? (p->P < 2 || p->rank < 0 || p->rank >= p->P) : p->rank != 0)
    return CSBP_ERR_INVALID;
  if (p->d != 64 && p->d != 128) return CSBP_ERR_UNSUPPORTED;
  if (p->tile_q != p->tile_kv) return CSBP_ERR_UNSUPPORTED;
  // No tensor of the problem reaches 2^39 elements (1 TiB of bf16, beyond any
  // one GPU), so every element and byte count below stays well inside int64.
  // Tested by division so that no product can overflow.
  constexpr int64_t kMaxElems = int64_t(1) << 39;
  const int64_t rows = static_cast<int64_t>(p->batch) * p->L;  // < 2^62
  if (rows >= kMaxElems || p->Hq > (kMaxElems - 1) / rows ||
      p->d > (kMaxElems - 1) / (rows * p->Hq))
    return CSBP_ERR_UNSUPPORTED;
  if (p->P > 1) {
    const int64_t B = p->L / p->M;
    if (B % (2 * p->P) != 0) return CSBP_ERR_UNSUPPORTED;
    if ((p->L / (2 * p->P)) % p->tile_kv != 0) return CSBP_ERR_UNSUPPORTED;
    if (p->P + 1 > kMaxParts) return CSBP_ERR_UNSUPPORTED;
  }
  return CSBP_OK;
}

// FNV-1a over the problem fields a work list depends on (batch, heads, d and
// the scale do not change it): lets the attention entry points refuse a list
// built for another problem.
uint64_t schedule_key(const csbp_problem* p) {
  const int32_t f[11] = {p->L, p->M, p->tile_q, p->tile_kv, p->P, p->has_clean_queries,
                         p->window, p->clean_causal, p->bwd_chunk, p->per_rank, p->rank};
  uint64_t h = 1469598103934665603ull;
  for (int32_t v : f) {
    for (int b = 0; b < 4; ++b) {
      h ^= static_cast<uint64_t>((static_cast<uint32_t>(v) >> (8 * b)) & 0xffu);
      h *= 1099511628211ull;
    }
  }
  return h;
}

int64_t bwd_chunk_tiles(const csbp_problem* p) { return p->bwd_chunk; }

bool bwd_windowed(const csbp_problem* p) {
  const int64_t nT = (static_cast<int64_t>(p->L) + p->tile_q - 1) / p->tile_q;
  return p->bwd_chunk > 0 && nT > p->bwd_chunk;
}

}  // namespace csbp

using namespace csbp;

extern "C" csbp_status csbp_block_schedule(const csbp_problem* problem, int32_t* block_owner,
                                           int32_t* chunk_owner, void* work, int64_t work_cap,
                                           csbp_schedule_info* info) {
  csbp_status st = validate_problem(problem);
  if (st != CSBP_OK) return st;
  if (!info) return CSBP_ERR_INVALID;
  const int64_t L = problem->L, M = problem->M, T = problem->tile_q;
  const int32_t P = problem->P;
  const int64_t B = L / M;
  const int64_t nT = (L + T - 1) / T;
  if (nT > (int64_t)1 << 30) return CSBP_ERR_UNSUPPORTED;
  const int64_t W = problem->window;
  const bool causal = problem->clean_causal != 0;
  auto classify = [&](int qs, int64_t qt, int ks, int64_t kt) {
    return (W > 0 || causal) ? classify_tile_ranges(qs, qt, ks, kt, L, M, T, W, causal)
                             : classify_tile(qs, qt, ks, kt, L, M, T);
  };

  // ---- ownership (P == 1: one shard owning both chunks)
  std::vector<int32_t> co(2 * P);
  for (int32_t r = 0; r < P; ++r) {
    co[r] = r;
    co[2 * P - 1 - r] = r;
  }
  const int64_t chunk_len = (P > 1) ? L / (2 * P) : 0;
  auto clean_part = [&](int64_t pos) -> int32_t {
    if (P == 1) return 0;
    return co[pos / chunk_len];
  };
  if (chunk_owner) std::memcpy(chunk_owner, co.data(), sizeof(int32_t) * 2 * P);
  if (block_owner) {
    for (int64_t b = 0; b < B; ++b) {
      if (P == 1) {
        block_owner[b] = 0;
      } else {
        block_owner[b] = co[(b * M) / chunk_len];
      }
    }
  }

  // ---- the query tiles this list covers: all, or (per_rank) those of the
  //      two clean chunks the rank owns, in both copies (a chunk is a whole
  //      number of tiles and of blocks, so a tile lies in one chunk and its
  //      corrupted blocks belong to that chunk's owner)
  const bool per_rank = problem->per_rank != 0;
  auto owned_tile = [&](int64_t qt) {
    return !per_rank || co[(qt * T) / chunk_len] == problem->rank;
  };

  // ---- forward tasks: per query tile (P == 1 or per_rank, fused) or per
  //      (tile, part)
  const int n_qs = problem->has_clean_queries ? 2 : 1;
  const int q_stream0 = problem->has_clean_queries ? 0 : 1;
  std::vector<Task> fwd;
  int64_t pairs = 0;
  for (int qs = q_stream0; qs < 2; ++qs) {
    for (int64_t qt = 0; qt < nT; ++qt) {
      if (!owned_tile(qt)) continue;
      std::vector<Seg> segs;
      std::vector<int32_t> seg_part;
      for (int ks = 0; ks < 2; ++ks) {
        int64_t ka, kb;
        tile_span([&](int64_t i, int64_t& lo, int64_t& hi) {
                    key_range(qs, ks, i, L, M, W, causal, lo, hi);
                  },
                  qt, L, T, ka, kb);
        for (int64_t kt = ka; kt < kb; ++kt) {
          const int cls = classify(qs, qt, ks, kt);
          if (!cls) continue;
          ++pairs;
          const int32_t part = (ks == 1) ? P : clean_part(kt * T);
          push_tile(segs, seg_part, ks, (int32_t)kt, cls, part);
        }
      }
      if (P == 1 || per_rank) {
        Task t{qs, (int32_t)qt, -1, segs, 0, 0};
        for (auto& s : segs) t.cost += s.end - s.begin;
        t.canon = W > 0 ? (int64_t)qt * 2 + qs : ((int64_t)qs * nT + qt);
        fwd.push_back(std::move(t));
      } else {
        for (int32_t part = 0; part <= P; ++part) {
          Task t{qs, (int32_t)qt, part, {}, 0, 0};
          for (size_t i = 0; i < segs.size(); ++i)
            if (seg_part[i] == part) {
              t.segs.push_back(segs[i]);
              t.cost += segs[i].end - segs[i].begin;
            }
          if (t.segs.empty()) continue;
          // equal-cost tasks of one part and copy sit next to each other, so
          // the two query tiles a forward CTA pairs share their key tiles
          t.canon = W > 0 ? ((int64_t)part * nT + qt) * 2 + qs : ((int64_t)part * 2 + qs) * nT + qt;
          fwd.push_back(std::move(t));
        }
      }
    }
  }
  (void)n_qs;

  // ---- backward tasks: per key tile, segments over query tiles (per key
  //      tile and query-tile window when the ranges are long)
  const bool windowed = bwd_windowed(problem);
  const int64_t chunk = bwd_chunk_tiles(problem);
  std::vector<Task> bwd;
  for (int ks = 0; ks < 2; ++ks) {
    for (int64_t kt = 0; kt < nT; ++kt) {
      Task t{ks, (int32_t)kt, (ks == 1) ? P : clean_part(kt * T), {}, 0, 0};
      std::vector<int32_t> dummy_part;
      for (int qs = q_stream0; qs < 2; ++qs) {
        int64_t qa, qb;
        tile_span([&](int64_t j, int64_t& lo, int64_t& hi) {
                    query_range(qs, ks, j, L, M, W, causal, lo, hi);
                  },
                  kt, L, T, qa, qb);
        for (int64_t qt = qa; qt < qb; ++qt) {
          if (!owned_tile(qt)) continue;
          const int cls = classify(qs, qt, ks, kt);
          if (!cls) continue;
          push_tile(t.segs, dummy_part, qs, (int32_t)qt, cls, 0);
          t.cost += 1;
        }
      }
      // emitted even when no query reads the tile: its dK/dV are then zero
      t.canon = (int64_t)ks * nT + kt;
      if (!windowed || t.segs.empty()) {
        t.flags = windowed ? 1 : 0;
        bwd.push_back(std::move(t));
        continue;
      }
      // one task per window of `chunk` query tiles, counted from the last
      // tile, so the CTAs of a wave walk the same window in step and share
      // its Q / dO tiles and dQ rows in L2 however long the whole range is
      for (int32_t j = 0;; ++j) {
        const int64_t hi = nT - (int64_t)j * chunk;
        if (hi <= 0) break;
        const int64_t lo = hi - chunk > 0 ? hi - chunk : 0;
        Task u{t.a_stream, t.a_tile, t.part, {}, 0, t.canon, 1, j};
        for (const Seg& g : t.segs) {
          const int64_t b = g.begin > lo ? g.begin : lo;
          const int64_t e = g.end < hi ? g.end : hi;
          if (b >= e) continue;
          u.segs.push_back({g.stream, (int32_t)b, (int32_t)e, g.flags});
          u.cost += (int32_t)(e - b);
        }
        if (!u.segs.empty()) bwd.push_back(std::move(u));
      }
    }
  }

  auto heavy_first = [](const Task& a, const Task& b) {
    if (a.window != b.window) return a.window < b.window;
    if (a.cost != b.cost) return a.cost > b.cost;
    return a.canon < b.canon;
  };
  // With a sliding window every query tile reads about the same number of
  // key tiles, and the clean and the corrupted tile at one position read the
  // same window of clean keys: forward tasks then run in (part, tile, copy)
  // order, so a CTA's two tasks are that pair and its walk wastes one tile
  // in twenty, where cost order would pair two corrupted (or two clean)
  // neighbours.  Otherwise heaviest first.
  if (W > 0)
    std::sort(fwd.begin(), fwd.end(), [](const Task& a, const Task& b) { return a.canon < b.canon; });
  else
    std::sort(fwd.begin(), fwd.end(), heavy_first);
  std::sort(bwd.begin(), bwd.end(), heavy_first);

  int64_t n_fseg = 0, n_bseg = 0;
  for (auto& t : fwd) n_fseg += (int64_t)t.segs.size();
  for (auto& t : bwd) n_bseg += (int64_t)t.segs.size();
  const int64_t off_ft = kHeaderWords;
  const int64_t off_fs = off_ft + (int64_t)fwd.size() * kTaskWords;
  const int64_t off_bt = off_fs + n_fseg * kSegWords;
  const int64_t off_bs = off_bt + (int64_t)bwd.size() * kTaskWords;
  const int64_t total = off_bs + n_bseg * kSegWords;
  if (total > INT32_MAX) return CSBP_ERR_UNSUPPORTED;

  info->n_fwd_tasks = (int32_t)fwd.size();
  info->n_fwd_segments = (int32_t)n_fseg;
  info->n_bwd_tasks = (int32_t)bwd.size();
  info->n_bwd_segments = (int32_t)n_bseg;
  info->tile_pairs = pairs;
  info->bytes = total * (int64_t)sizeof(int32_t);
  info->problem_key = schedule_key(problem);
  if (!work || work_cap < info->bytes) return CSBP_ERR_CAPACITY;

  int32_t* w = static_cast<int32_t*>(work);
  std::memset(w, 0, (size_t)info->bytes);
  const int32_t hdr[kHeaderWords] = {kMagic,
                                     kVersion,
                                     problem->L,
                                     problem->M,
                                     (int32_t)T,
                                     P,
                                     problem->has_clean_queries,
                                     (int32_t)fwd.size(),
                                     (int32_t)n_fseg,
                                     (int32_t)bwd.size(),
                                     (int32_t)n_bseg,
                                     (int32_t)off_ft,
                                     (int32_t)off_fs,
                                     (int32_t)off_bt,
                                     (int32_t)off_bs,
                                     (int32_t)total};
  std::memcpy(w, hdr, sizeof(hdr));
  auto emit = [&](const std::vector<Task>& tasks, int64_t off_task, int64_t off_seg) {
    int64_t s = 0;
    for (size_t i = 0; i < tasks.size(); ++i) {
      const Task& t = tasks[i];
      int32_t* tw = w + off_task + (int64_t)i * kTaskWords;
      tw[0] = t.a_stream;
      tw[1] = t.a_tile;
      tw[2] = t.part;
      tw[3] = (int32_t)s;
      tw[4] = (int32_t)t.segs.size();
      tw[5] = t.cost;
      tw[6] = t.flags;
      tw[7] = t.window;
      for (const Seg& g : t.segs) {
        int32_t* sw = w + off_seg + s * kSegWords;
        sw[0] = g.stream;
        sw[1] = g.begin;
        sw[2] = g.end;
        sw[3] = g.flags;
        ++s;
      }
    }
  };
  emit(fwd, off_ft, off_fs);
  emit(bwd, off_bt, off_bs);
  return CSBP_OK;
}
