// la_api.cu -- the C ABI of lean_attn.h: host tile planner, schedule
// upload, argument checks and kernel launches.
//
// Planner rules (xllm-io paper review of LeanAttention):
//   "3.3 LeanTile"              T = 256 tokens at d = 64, 128 at d = 128
//                               (other head dims: the tile that keeps a
//                               stage near 64 KiB of K+V, see default_tile)
//   "3.4 stream-K decomposition" tiles of all units on one line, split
//                               evenly over G CTAs, crossing unit boundaries
//   "3.5 execution flow"        I_G = I / G per CTA; host and finishing CTA
//                               per output tile; non-host CTAs hand their
//                               partial to the host through global memory
//   "4.3 work distribution"     fixed partitions (FlashAttention-2,
//                               FlashDecoding) for the baselines
// The planner walks CTA ranges arithmetically in O(G + units).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "la_internal.h"
#include "la_schedule.h"
#include "lean_attn.h"

namespace {

constexpr int kMaxGrid = 1 << 20;

// Query rows per unit head the kernel instance holds: rows rounded up to 1,
// 2, 4, 8 or 16 (the spare rows are zero queries that are never written
// out); more than 16 rows run on the tcgen05 kernel's 128-row instance.
int instance_rows(int rows) {
  return rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : rows <= 8 ? 8 : rows <= 16 ? 16 : la::kWideRows;
}

// Query rows one unit can hold at head dim d: where the tcgen05 kernel is
// built, 128 (64 at d = 256); else 16.
int max_unit_rows(int d) { return la::wide_supported(d) ? la::wide_max_rows(d) : 16; }

// Query blocks per kv head: the fewest blocks of equal size (a divisor of
// grp) whose grp / qb * nq query rows fit one unit; 0 when none does (nq
// alone is more than a unit holds).
int query_blocks(int grp, int nq, int d) {
  const int lim = max_unit_rows(d);
  if (grp < 1 || nq < 1 || nq > lim) return 0;
  for (int qb = 1; qb <= grp; ++qb)
    if (grp % qb == 0 && (grp / qb) * nq <= lim) return qb;
  return 0;
}

// Query rows of one unit head (a kv head, or one query block of one).
int unit_rows(int grp, int nq, int d) {
  const int qb = query_blocks(grp, nq, d);
  return qb == 0 ? 0 : (grp / qb) * nq;
}

// LeanTile tokens a unit of `rows` query rows uses by default: 128 on the
// tcgen05 kernel (64 at d = 256); else slab_tile for stream-K schedules and
// the table's size for fixed partitions.
int unit_tile(int d, int rows, int kind) {
  if (rows > 16) return la::wide_tile(d);
  return kind == 0 ? la::slab_tile(d, rows) : la::default_tile(d);
}

// Whether (d, T, hp) is built for units of `rows` query rows.
bool unit_tile_supported(int d, int T, int hp, int rows) {
  if (rows > 16) return la::wide_supported(d) && T == la::wide_tile(d) && hp == 1;
  return la::tile_supported(d, T, hp);
}

la_status check_shape(int batch, int hq, int hkv, int d, const int32_t* cu) {
  if (batch <= 0 || hq <= 0 || hkv <= 0 || cu == nullptr) return LA_ERR_INVALID;
  if (hq % hkv != 0) return LA_ERR_INVALID;
  if (cu[0] != 0) return LA_ERR_INVALID;
  for (int b = 0; b < batch; ++b)
    if (cu[b + 1] <= cu[b]) return LA_ERR_INVALID;  // every context holds >= 1 token
  if (d <= 0) return LA_ERR_INVALID;
  if (la::default_tile(d) == 0) return LA_ERR_UNSUPPORTED;
  // element offsets are formed in 64 bits, tile indices in 32 bits
  if ((int64_t)hkv * cu[batch] > (int64_t)INT32_MAX * 64) return LA_ERR_UNSUPPORTED;
  return LA_OK;
}

// Units (b, group of hp kv heads or one query block of a kv head) in
// request-major order and their tile prefix sums.
bool build_units(la_schedule* s) {
  const int groups = s->unit_heads() / s->hp;
  s->U = s->batch * groups;
  s->unit_iter.assign((size_t)s->U + 1, 0);
  int64_t acc = 0;
  for (int b = 0; b < s->batch; ++b) {
    const int64_t L = (int64_t)s->cu[b + 1] - s->cu[b];
    const int64_t tiles = (L + s->T - 1) / s->T;
    for (int h = 0; h < groups; ++h) {
      s->unit_iter[(size_t)b * groups + h] = (int32_t)acc;
      acc += tiles;
      if (acc > INT32_MAX) return false;
    }
  }
  s->unit_iter[s->U] = (int32_t)acc;
  s->I = acc;
  return true;
}

void add_seg(la_schedule* s, int unit, int t0, int t1, int kind, int peer) {
  s->segs.insert(s->segs.end(), {unit, t0, t1, kind, peer});
}

// CTA of global iteration i under the even split of I over G.
int cta_of(int64_t i, int64_t I, int G) {
  const int64_t q = I / G, r = I % G;
  if (q == 0 || i < r * (q + 1)) return (int)(i / (q + 1));
  return (int)(r + (i - r * (q + 1)) / q);
}

la_status plan_lean(la_schedule* s) {
  const int G = s->G;
  const int64_t I = s->I, q = I / G, r = I % G;
  s->cta_iter.resize((size_t)G + 1);
  for (int g = 0; g <= G; ++g) s->cta_iter[g] = (int32_t)(g * q + std::min<int64_t>(g, r));
  s->unit_host.resize(s->U);
  s->unit_fin.resize(s->U);
  for (int u = 0; u < s->U; ++u) {
    s->unit_host[u] = cta_of(s->unit_iter[u], I, G);
    s->unit_fin[u] = cta_of((int64_t)s->unit_iter[u + 1] - 1, I, G);
  }
  s->cta_seg.assign((size_t)G + 1, 0);
  s->segs.clear();
  int u = 0;
  for (int g = 0; g < G; ++g) {
    s->cta_seg[g] = (int32_t)(s->segs.size() / la::kSegWords);
    int64_t i = s->cta_iter[g];
    const int64_t e = s->cta_iter[g + 1];
    while (i < e) {
      while (s->unit_iter[u + 1] <= i) ++u;
      const int64_t ub = s->unit_iter[u], ue = s->unit_iter[u + 1];
      const int64_t j = std::min(e, ue);
      const int t0 = (int)(i - ub), t1 = (int)(j - ub);
      if (i == ub && j == ue)
        add_seg(s, u, t0, t1, la::kWhole, -1);
      else if (i == ub)
        add_seg(s, u, t0, t1, la::kHost, s->unit_fin[u]);
      else
        add_seg(s, u, t0, t1, la::kNonHost, -1);
      i = j;
    }
  }
  s->cta_seg[G] = (int32_t)(s->segs.size() / la::kSegWords);
  return LA_OK;
}

la_status plan_fixed(la_schedule* s) {
  s->cta_iter.assign(1, 0);
  s->cta_seg.assign(1, 0);
  s->segs.clear();
  s->unit_host.resize(s->U);
  s->unit_fin.resize(s->U);
  int g = 0;
  for (int u = 0; u < s->U; ++u) {
    const int64_t n = (int64_t)s->unit_iter[u + 1] - s->unit_iter[u];
    const int64_t k = std::min<int64_t>(s->splits, n);
    s->unit_host[u] = g;
    for (int64_t p = 0; p < k; ++p) {
      const int t0 = (int)(p * n / k), t1 = (int)((p + 1) * n / k);
      add_seg(s, u, t0, t1, k == 1 ? la::kWhole : la::kPartial, -1);
      s->cta_iter.push_back(s->cta_iter.back() + (t1 - t0));
      s->cta_seg.push_back((int32_t)(s->segs.size() / la::kSegWords));
      if (++g > kMaxGrid) return LA_ERR_UNSUPPORTED;
    }
    s->unit_fin[u] = g - 1;
  }
  s->G = g;
  return LA_OK;
}

// Device segment records: the planner's words plus L and the slab's first row
// (and, for a piece of a split unit, its finisher and host CTAs).
void build_dev_segs(la_schedule* s) {
  const size_t n = s->segs.size() / la::kSegWords;
  s->dev_segs.assign(n * la::kDevSegWords, 0);
  for (size_t i = 0; i < n; ++i) {
    const int32_t* sg = &s->segs[i * la::kSegWords];
    int32_t* dv = &s->dev_segs[i * la::kDevSegWords];
    const int groups = s->unit_heads() / s->hp;
    // first kv head of the unit (the kv head of its query block)
    const int b = sg[0] / groups, kvh = (sg[0] % groups) * s->hp / s->qb;
    const int64_t L = (int64_t)s->cu[b + 1] - s->cu[b];
    const int64_t row0 = (int64_t)s->hkv * s->cu[b] + (int64_t)kvh * L;
    for (int w = 0; w < la::kSegWords; ++w) dv[w] = sg[w];
    dv[5] = (int32_t)L;
    dv[6] = (int32_t)(uint32_t)(row0 & 0xffffffffLL);
    dv[7] = (int32_t)(row0 >> 32);
    dv[8] = s->cu[b];
    dv[9] = b;
    dv[10] = kvh;
    dv[11] = 0;
    if (sg[3] == la::kHost || sg[3] == la::kNonHost) {  // a piece of a split unit: its host and finisher CTAs
      dv[4] = s->unit_fin[sg[0]];
      dv[11] = s->unit_host[sg[0]];
    }
  }
}

la_status make_schedule(int batch, int hq, int hkv, int d, const int32_t* cu, int kind, int grid_or_splits,
                        la_schedule** out, int tile = 0, int hp = 1, int nq = 1) {
  if (out == nullptr) return LA_ERR_INVALID;
  *out = nullptr;
  const la_status st = check_shape(batch, hq, hkv, d, cu);
  if (st != LA_OK) return st;
  if (hp < 1 || hkv % hp != 0) return LA_ERR_INVALID;
  const int qb = query_blocks(hq / hkv, nq, d);
  if (qb == 0) return LA_ERR_UNSUPPORTED;
  const int rows = (hq / hkv / qb) * nq;
  // units are counted in 32 bits (and index q rows with their query heads)
  if ((int64_t)batch * hkv * qb > (int64_t)INT32_MAX / 16 || (int64_t)batch * nq * hq > (int64_t)INT32_MAX / 16)
    return LA_ERR_UNSUPPORTED;
  // a query block, or a unit of more than 16 rows, is one kv head
  if ((qb > 1 || rows > 16) && hp != 1) return LA_ERR_UNSUPPORTED;
  // stream-K on the slab layout: slab_tile; the fixed partitions keep the
  // table's tile (with few busy SMs each CTA needs the deeper 192 KiB ring)
  if (tile == 0) tile = hp == 1 ? unit_tile(d, rows, kind) : la::default_tile(d) / hp;
  if (tile < 0) return LA_ERR_INVALID;
  if (!unit_tile_supported(d, tile, hp, rows)) return LA_ERR_UNSUPPORTED;
  la_schedule* s = new (std::nothrow) la_schedule();
  if (s == nullptr) return LA_ERR_INVALID;
  s->serial = la_next_schedule_serial();
  s->batch = batch;
  s->hq = hq;
  s->hkv = hkv;
  s->d = d;
  s->grp = hq / hkv;
  s->nq = nq;
  s->qb = qb;
  s->R = instance_rows(rows);
  s->hp = hp;
  s->T = tile;
  s->kind = kind;
  s->cu.assign(cu, cu + batch + 1);
  if (!build_units(s)) {
    delete s;
    return LA_ERR_UNSUPPORTED;
  }
  la_status r;
  if (kind == 0) {
    s->G = grid_or_splits;
    r = plan_lean(s);
  } else {
    s->splits = grid_or_splits;
    r = plan_fixed(s);
  }
  if (r != LA_OK) {
    delete s;
    return r;
  }
  build_dev_segs(s);
  *out = s;
  return LA_OK;
}

// CTAs per SM of the decode kernel, cached per (device, d, T, grp, hp).
la_status capacity(int d, int T, int grp, int* per_sm, int hp = 1) {
  static std::mutex mu;
  static std::map<long long, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  const long long key = ((((long long)dev * 1024 + d) * 1024 + T) * 256 + grp) * 16 + hp;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *per_sm = it->second;
    return LA_OK;
  }
  cudaError_t e = la::decode_capacity(d, T, grp, hp, per_sm);
  if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return LA_ERR_CUDA;
  cache[key] = *per_sm;
  return LA_OK;
}

la_status device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LA_ERR_CUDA;
  return LA_OK;
}

// Upload the schedule tables to the current device once.
la_status ensure_uploaded(la_schedule* s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(s->mu);
  if (s->dev != nullptr) return s->device == dev ? LA_OK : LA_ERR_INVALID;
  std::vector<int32_t> buf;
  s->off_cu = buf.size();
  buf.insert(buf.end(), s->cu.begin(), s->cu.end());
  s->off_cta_seg = buf.size();
  buf.insert(buf.end(), s->cta_seg.begin(), s->cta_seg.end());
  while (buf.size() % 4 != 0) buf.push_back(0);  // segment records are read as 16-byte vectors
  s->off_segs = buf.size();
  buf.insert(buf.end(), s->dev_segs.begin(), s->dev_segs.end());
  s->off_host = buf.size();
  buf.insert(buf.end(), s->unit_host.begin(), s->unit_host.end());
  s->off_fin = buf.size();
  buf.insert(buf.end(), s->unit_fin.begin(), s->unit_fin.end());
  int32_t* d = nullptr;
  if (cudaMalloc(&d, buf.size() * sizeof(int32_t)) != cudaSuccess) return LA_ERR_CUDA;
  if (cudaMemcpy(d, buf.data(), buf.size() * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(d);
    return LA_ERR_CUDA;
  }
  s->dev = d;
  s->device = dev;
  return LA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- shape-driven choice among the three partitions ----------------------
// Time model (seconds) of a launch whose CTAs each stream a fixed number of
// bytes: CTAs are dispatched in order onto `slots` SMs as SMs free up (the
// hardware's in-order block dispatch); while n CTAs run, together they read
// R(n) = r_max * (1 - exp(-n / n0)) bytes/s, shared equally. Jobs finish in
// order of their cumulative progress, so a heap of finish thresholds gives
// the makespan. cap > 0 bounds the rate of one CTA (a kernel whose tile
// loop, not HBM, limits a lone CTA).
double simulate_dispatch(const std::vector<double>& job_bytes, int slots, double r_max, double n0,
                         double cap = 0.0) {
  if (job_bytes.empty()) return 0.0;
  std::vector<double> heap;  // min-heap of progress thresholds of running jobs
  auto cmp = [](double a, double b) { return a > b; };
  size_t next = 0;
  double progress = 0.0, t = 0.0;
  while (next < job_bytes.size() && (int)heap.size() < slots) {
    heap.push_back(progress + job_bytes[next++]);
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  while (!heap.empty()) {
    const double n = (double)heap.size();
    double rate = r_max * (1.0 - std::exp(-n / n0)) / n;
    if (cap > 0.0) rate = std::min(rate, cap);
    std::pop_heap(heap.begin(), heap.end(), cmp);
    const double thr = heap.back();
    heap.pop_back();
    t += (thr - progress) / rate;
    progress = thr;
    if (next < job_bytes.size()) {
      heap.push_back(progress + job_bytes[next++]);
      std::push_heap(heap.begin(), heap.end(), cmp);
    }
  }
  return t;
}

// Bytes of K+V of tiles [t0, t1) of unit u.
double piece_bytes(const la_schedule* s, int u, int t0, int t1) {
  const int b = u / (s->unit_heads() / s->hp);
  const int64_t L = (int64_t)s->cu[b + 1] - s->cu[b];
  const int64_t tok = std::min<int64_t>((int64_t)t1 * s->T, L) - (int64_t)t0 * s->T;
  return (double)tok * s->hp * s->d * 2.0 * 2.0;
}

// Predicted time of a schedule: per-CTA byte totals through the dispatch model,
// a start-up latency for every CTA an SM runs in turn (its first tile must
// arrive before it computes), the host CTAs' merge when units are split
// within the launch, and launch overheads (two launches for fixed splits > 1).
// Constants fitted to GB300 measurements: aggregate read rate with n busy SMs
// 7.5 TB/s * (1 - exp(-n / 60)) (3.1 TB/s at 32, 6.6 at 128, 6.9 at 152);
// 3 us from CTA start to its first tile; 2.5 us for a host CTA's merge on
// the 16-row kernel.
double predict_seconds(const la_schedule* s, int slots) {
  constexpr double kRateMax = 7.5e12, kRateN0 = 60.0;
  constexpr double kLaunch = 8e-6, kMergeLaunch = 4e-6, kStartup = 3e-6, kHostMerge = 2.5e-6;
  // the tcgen05 kernel's merge of a split unit, shared by the unit's CTAs:
  // about 3 us plus 0.11 us per piece of the unit (GB300: 10 pieces of 64
  // rows at d = 128 ~4 us after the last piece; 152 pieces ~20 us)
  constexpr double kWideMerge = 3e-6, kWideMergePerPiece = 0.11e-6;
  // the fixed split's merge launch for tcgen05 records: 0.13 us per piece of
  // a unit (152 pieces of 64 rows at d = 128: 64 us in all, 21 of them the
  // pieces' tile loops)
  constexpr double kWideCombinePerPiece = 0.13e-6;
  std::vector<double> jobs((size_t)s->G, 0.0);
  bool split = false;
  int max_peers = 0;
  for (int g = 0; g < s->G; ++g)
    for (int i = s->cta_seg[g]; i < s->cta_seg[g + 1]; ++i) {
      const int32_t* sg = &s->segs[(size_t)i * la::kSegWords];
      jobs[g] += piece_bytes(s, sg[0], sg[1], sg[2]);
      if (sg[3] == la::kHost) {
        split = true;
        max_peers = std::max(max_peers, sg[4] - g);
      }
    }
  const int rounds = (s->G + slots - 1) / std::max(1, slots);  // CTAs one SM runs in turn
  // a CTA of the tcgen05 kernel streams one 128-token tile per 1.55 us at
  // most (its softmax and MMA chain), whatever HBM could give it
  const double cap = s->R == la::kWideRows ? (double)s->T * s->d * 4.0 / 1.55e-6 : 0.0;
  double t = simulate_dispatch(jobs, slots, kRateMax, kRateN0, cap) + kLaunch + kStartup * rounds;
  if (split) t += s->R == la::kWideRows ? kWideMerge + kWideMergePerPiece * (max_peers + 1) : kHostMerge;
  if (s->kind == 1 && s->splits > 1) {
    t += kMergeLaunch;
    if (s->R == la::kWideRows) {  // the tcgen05 records' merge reads each row's pieces one after another
      int most = 1;
      for (int u = 0; u < s->U; ++u) most = std::max(most, s->unit_fin[u] - s->unit_host[u] + 1);
      t += kWideCombinePerPiece * most;
    }
  }
  return t;
}

}  // namespace

namespace la {

int cached_capacity(int d, int T, int grp, int hp, int* per_sm) { return capacity(d, T, grp, per_sm, hp); }



int device_sm_count(int* sms) { return device_sms(sms); }

int slab_tile(int d, int rows) { return (d == 128 && rows <= 2) ? 64 : default_tile(d); }

int stream_stages(int d, int T, int hp, int kv_layout) {
  // Measured on one GB300 (us per call, library default vs the whole ring):
  // d 96, 48 KiB stages: 3 of 4 (slab 229.5 vs 232.7; token-major with 4
  // kv heads per unit 239.3 vs 243.2); d 128 with 128-token tiles: 2 of 3
  // (GQA d128 55.4 vs 59.2, at batch 1 35.2 vs 37.1; paged 16-token pages
  // 164.7 vs 172.7), except token-major caches (161.4 vs 159.0 with 3).
  if (d == 96 && T * hp == 128) return 3;
  if (d == 128 && T == 128 && hp == 1 && kv_layout != kKvTokenMajor) return 2;
  return 0;
}

int default_tile(int d) {
  switch (d) {
    case 64: return 256;   // the review's LeanTile table
    case 128: return 128;  // the review's LeanTile table
    case 80: return 128;   // 40 KiB of K+V per tile
    case 96: return 128;   // 48 KiB
    case 256: return 64;   // 64 KiB, like the table's two sizes
    default: return 0;
  }
}

bool tile_supported(int d, int T, int hp) {
  // units of several kv heads: the default tile of the head dim divided over
  // the heads (the tile keeps its bytes)
  if (hp > 1) {
    const bool built = (d == 64 && hp == 2) || (d == 80 && (hp == 2 || hp == 8)) ||
                       (d == 96 && (hp == 2 || hp == 4));
    return built && T * hp == default_tile(d);
  }
  if (hp != 1) return false;
  switch (d) {
    case 64: return T == 256 || T == 128;
    case 128: return T == 128 || T == 64;
    case 80:
    case 96: return T == 128;
    case 256: return T == 64;
    default: return false;
  }
}

cudaError_t launch_decode(int d, int T, int grp, int hp, int dtype, const KParams& p, cudaStream_t st) {
  if (grp == kWideRows) return (hp == 1 && T == wide_tile(d)) ? launch_wide(d, dtype, p, st) : cudaErrorInvalidValue;
  switch (d * 16 + hp) {
    case 64 * 16 + 2: return launch_decode_d64_hp2(T, grp, dtype, p, st);
    case 80 * 16 + 2: return launch_decode_d80_hp2(T, grp, dtype, p, st);
    case 80 * 16 + 8: return launch_decode_d80_hp8(T, grp, dtype, p, st);
    case 96 * 16 + 2: return launch_decode_d96_hp2(T, grp, dtype, p, st);
    case 96 * 16 + 4: return launch_decode_d96_hp4(T, grp, dtype, p, st);
    default: break;
  }
  if (hp != 1) return cudaErrorInvalidValue;
  switch (d) {
    case 64: return launch_decode_d64(T, grp, dtype, p, st);
    case 80: return launch_decode_d80(T, grp, dtype, p, st);
    case 96: return launch_decode_d96(T, grp, dtype, p, st);
    case 128: return launch_decode_d128(T, grp, dtype, p, st);
    case 256: return launch_decode_d256(T, grp, dtype, p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(int d, int grp, const CParams& p, cudaStream_t st) {
  if (grp == kWideRows) return launch_combine_wide(d, p, st);
  switch (d) {
    case 64: return launch_combine_d64(grp, p, st);
    case 80: return launch_combine_d80(grp, p, st);
    case 96: return launch_combine_d96(grp, p, st);
    case 128: return launch_combine_d128(grp, p, st);
    case 256: return launch_combine_d256(grp, p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t decode_capacity(int d, int T, int grp, int hp, int* per_sm) {
  if (grp == kWideRows) return (hp == 1 && T == wide_tile(d)) ? wide_capacity(d, per_sm) : cudaErrorInvalidValue;
  switch (d * 16 + hp) {
    case 64 * 16 + 2: return decode_capacity_d64_hp2(T, grp, per_sm);
    case 80 * 16 + 2: return decode_capacity_d80_hp2(T, grp, per_sm);
    case 80 * 16 + 8: return decode_capacity_d80_hp8(T, grp, per_sm);
    case 96 * 16 + 2: return decode_capacity_d96_hp2(T, grp, per_sm);
    case 96 * 16 + 4: return decode_capacity_d96_hp4(T, grp, per_sm);
    default: break;
  }
  if (hp != 1) return cudaErrorInvalidValue;
  switch (d) {
    case 64: return decode_capacity_d64(T, grp, per_sm);
    case 80: return decode_capacity_d80(T, grp, per_sm);
    case 96: return decode_capacity_d96(T, grp, per_sm);
    case 128: return decode_capacity_d128(T, grp, per_sm);
    case 256: return decode_capacity_d256(T, grp, per_sm);
    default: return cudaErrorInvalidValue;
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up once.
EncodeTiled encode_fn() {
  static std::mutex mu;
  static EncodeTiled fn = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

cudaError_t encode_kv_maps(const void* k, const void* v, long long rows, int d, int T, int W, int elem_type,
                           CUtensorMap* mk, CUtensorMap* mv) {
  const EncodeTiled fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  if (rows <= 0 || rows > (1LL << 31) - 1) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)W, (cuuint32_t)T};
  const CUtensorMapSwizzle swz = W == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                          : (W == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = (CUtensorMapDataType)elem_type;
  for (int i = 0; i < 2; ++i) {
    CUresult r = fn(i == 0 ? mk : mv, dt, 2, const_cast<void*>(i == 0 ? k : v), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t encode_kv_maps_3d(const void* k, const void* v, long long rows, int hkv, int d, int bw, int hp,
                              int box_rows, bool swizzle, int elem_type, CUtensorMap* mk, CUtensorMap* mv) {
  const EncodeTiled fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  if (rows <= 0 || rows > (1LL << 31) - 1) return cudaErrorInvalidValue;
  if (hp < 1 || hkv % hp != 0) return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hkv * d * 2};
  const cuuint32_t box[3] = {(cuuint32_t)bw, (cuuint32_t)hp, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle)
    swz = bw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : (bw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  for (int i = 0; i < 2; ++i) {
    CUresult r = fn(i == 0 ? mk : mv, (CUtensorMapDataType)elem_type, 3, const_cast<void*>(i == 0 ? k : v), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace la

extern "C" {

la_status la_plan_ex(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                     int tile_tokens, la_schedule** out) {
  if (out != nullptr) *out = nullptr;
  int G = num_sms;
  if (G <= 0) {
    const la_status st = check_shape(batch, hq, hkv, d, cu_seqlens_k);
    if (st != LA_OK) return st;
    const int rows = unit_rows(hq / hkv, 1, d);
    const int T = tile_tokens == 0 ? unit_tile(d, rows, 0) : tile_tokens;
    if (T <= 0) return LA_ERR_INVALID;
    if (!unit_tile_supported(d, T, 1, rows)) return LA_ERR_UNSUPPORTED;
    int sms = 0, per_sm = 0;
    la_status e = device_sms(&sms);
    if (e != LA_OK) return e;
    e = capacity(d, T, instance_rows(rows), &per_sm);
    if (e != LA_OK) return e;
    G = sms * std::max(1, per_sm);
  }
  if (G > kMaxGrid) return LA_ERR_INVALID;
  return make_schedule(batch, hq, hkv, d, cu_seqlens_k, 0, G, out, tile_tokens);
}

la_status la_plan(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                  la_schedule** out) {
  return la_plan_ex(batch, hq, hkv, d, cu_seqlens_k, num_sms, 0, out);
}

la_status la_plan_spec(int batch, int hq, int hkv, int d, int nq, const int32_t* cu_seqlens_k, int num_sms,
                       la_schedule** out) {
  if (out != nullptr) *out = nullptr;
  la_status st = check_shape(batch, hq, hkv, d, cu_seqlens_k);
  if (st != LA_OK) return st;
  if (nq < 1) return LA_ERR_INVALID;
  const int rows = unit_rows(hq / hkv, nq, d);
  if (rows == 0) return LA_ERR_UNSUPPORTED;
  for (int b = 0; b < batch; ++b)
    if (cu_seqlens_k[b + 1] - cu_seqlens_k[b] < nq) return LA_ERR_INVALID;  // the query tokens are in the context
  const int R = instance_rows(rows);
  int G = num_sms;
  if (G <= 0) {
    int sms = 0, per_sm = 0;
    st = device_sms(&sms);
    if (st != LA_OK) return st;
    st = capacity(d, unit_tile(d, rows, 0), R, &per_sm);
    if (st != LA_OK) return st;
    G = sms * std::max(1, per_sm);
  }
  if (G > kMaxGrid) return LA_ERR_INVALID;
  return make_schedule(batch, hq, hkv, d, cu_seqlens_k, 0, G, out, 0, 1, nq);
}

la_status la_plan_kv(int batch, int hq, int hkv, int d, int nq, const int32_t* cu_seqlens_k, int heads_per_unit,
                     int tile_tokens, int num_sms, la_schedule** out) {
  if (out != nullptr) *out = nullptr;
  if (out == nullptr) return LA_ERR_INVALID;
  la_status st = check_shape(batch, hq, hkv, d, cu_seqlens_k);
  if (st != LA_OK) return st;
  if (nq < 1 || tile_tokens < 0) return LA_ERR_INVALID;
  int hp = heads_per_unit;
  const int rows = unit_rows(hq / hkv, nq, d);
  if (rows == 0) return LA_ERR_UNSUPPORTED;
  // more than 8 query rows per unit, or query blocks: units of one kv head only
  if (rows > 8 || query_blocks(hq / hkv, nq, d) > 1) {
    if (hp > 1) return LA_ERR_UNSUPPORTED;
    hp = 1;
  }
  if (hp == 0) {
    // the fewest kv heads whose rows together make whole 256-byte pieces
    // (d = 64: 2, 96: 4, 80: 8), else the most of those that divide hkv
    hp = 1;
    for (int h = 8; h >= 2; h /= 2)
      if ((h * d * 2) % 256 == 0 && hkv % h == 0 && la::tile_supported(d, la::default_tile(d) / h, h)) hp = h;
    if (hp == 1)
      for (int h = 8; h >= 2 && hp == 1; h /= 2)
        if (hkv % h == 0 && la::tile_supported(d, la::default_tile(d) / h, h)) hp = h;
  }
  if ((hp != 1 && hp != 2 && hp != 4 && hp != 8) || hkv % hp != 0) return LA_ERR_INVALID;
  for (int b = 0; b < batch; ++b)
    if (cu_seqlens_k[b + 1] - cu_seqlens_k[b] < nq) return LA_ERR_INVALID;  // the query tokens are in the context
  const int R = instance_rows(rows);
  const int T = tile_tokens != 0 ? tile_tokens : (rows > 16 ? la::wide_tile(d) : la::default_tile(d) / hp);
  if (!unit_tile_supported(d, T, hp, rows)) return LA_ERR_UNSUPPORTED;
  int G = num_sms;
  if (G <= 0) {
    int sms = 0, per_sm = 0;
    st = device_sms(&sms);
    if (st != LA_OK) return st;
    st = capacity(d, T, R, &per_sm, hp);
    if (st != LA_OK) return st;
    G = sms * std::max(1, per_sm);
  }
  if (G > kMaxGrid) return LA_ERR_INVALID;
  return make_schedule(batch, hq, hkv, d, cu_seqlens_k, 0, G, out, T, hp, nq);
}

la_status la_plan_fixed(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int splits,
                        la_schedule** out) {
  if (out != nullptr) *out = nullptr;
  if (splits <= 0) return LA_ERR_INVALID;
  return make_schedule(batch, hq, hkv, d, cu_seqlens_k, 1, splits, out);
}

la_status la_plan_auto(int batch, int hq, int hkv, int d, const int32_t* cu_seqlens_k, int num_sms,
                       la_schedule** out, double* predicted_us) {
  if (out != nullptr) *out = nullptr;
  if (out == nullptr) return LA_ERR_INVALID;
  la_status st = check_shape(batch, hq, hkv, d, cu_seqlens_k);
  if (st != LA_OK) return st;
  int slots = num_sms;
  if (slots <= 0) {
    int sms = 0, per_sm = 0;
    st = device_sms(&sms);
    if (st != LA_OK) return st;
    const int rows = unit_rows(hq / hkv, 1, d);
    if (rows == 0) return LA_ERR_UNSUPPORTED;
    st = capacity(d, unit_tile(d, rows, 0), instance_rows(rows), &per_sm);
    if (st != LA_OK) return st;
    slots = sms * std::max(1, per_sm);
  }
  la_schedule* cand[3] = {nullptr, nullptr, nullptr};
  st = make_schedule(batch, hq, hkv, d, cu_seqlens_k, 0, slots, &cand[0]);  // stream-K over every SM
  if (st == LA_OK) st = make_schedule(batch, hq, hkv, d, cu_seqlens_k, 1, 1, &cand[1]);  // one CTA per unit
  if (st == LA_OK) {
    const int units = cand[1]->U;
    const int k = std::max(2, (slots + units - 1) / units);  // fixed split that fills the SMs
    st = make_schedule(batch, hq, hkv, d, cu_seqlens_k, 1, k, &cand[2]);
  }
  if (st != LA_OK) {
    for (la_schedule* c : cand) delete c;
    return st;
  }
  int best = 0;
  double t[3];
  for (int i = 0; i < 3; ++i) {
    t[i] = predict_seconds(cand[i], slots);
    if (predicted_us != nullptr) predicted_us[i] = t[i] * 1e6;
    if (t[i] < t[best]) best = i;
  }
  for (int i = 0; i < 3; ++i)
    if (i != best) delete cand[i];
  *out = cand[best];
  return LA_OK;
}

int la_schedule_grid(const la_schedule* s) { return s ? s->G : -1; }

size_t la_workspace_size(const la_schedule* s) {
  if (s == nullptr) return 0;
  return la::workspace_bytes(s->G, s->d, s->R * s->hp);
}

la_status la_workspace_init(void* workspace, size_t bytes, la_stream_t stream) {
  if (workspace == nullptr || bytes < la::kHeaderBytes) return LA_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

la_status la_decode_kv(const void* q, const void* k, const void* v, la_dtype dt, const int32_t* cu_seqlens_k_dev,
                       const la_kv_desc* kv, const la_schedule* sc, void* workspace, void* out,
                       la_dtype_out out_dt, float scale, la_stream_t stream) {
  if (out_dt != LA_OUT_F32 && out_dt != LA_OUT_F16 && out_dt != LA_OUT_BF16) return LA_ERR_INVALID;
  const int out_dtype = (int)out_dt;
  if (kv == nullptr || sc == nullptr) return LA_ERR_INVALID;
  int kv_layout = la::kKvSlab, box_rows = 0, page_size = 0, bt_stride = 0;
  long long kv_rows = 0;
  if (kv->layout == LA_KV_TOKEN_MAJOR) {
    kv_layout = la::kKvTokenMajor;
    box_rows = sc->T;
    kv_rows = sc->cu[sc->batch];
  } else if (kv->layout == LA_KV_PAGED) {
    kv_layout = la::kKvPaged;
    page_size = kv->page_size;
    if (page_size < 16 || (page_size & (page_size - 1)) != 0 || kv->block_table == nullptr ||
        kv->num_pages <= 0 || !aligned(kv->block_table, 4))
      return LA_ERR_INVALID;
    if (kv->num_pages * (long long)page_size > (1LL << 31) - 1) return LA_ERR_UNSUPPORTED;
    int64_t need = 0;  // block-table entries the longest request uses
    for (int b = 0; b < sc->batch; ++b)
      need = std::max<int64_t>(need, ((int64_t)sc->cu[b + 1] - sc->cu[b] + page_size - 1) / page_size);
    if (kv->max_blocks < need) return LA_ERR_INVALID;
    bt_stride = kv->max_blocks;
    box_rows = std::min(sc->T, page_size);
    kv_rows = kv->num_pages * (long long)page_size;
  } else if (kv->layout != LA_KV_SLAB) {
    return LA_ERR_INVALID;
  }
  if (kv_layout == la::kKvSlab && sc->hp != 1) return LA_ERR_UNSUPPORTED;  // units of several heads: caches only
  if (kv_layout != la::kKvSlab) {
    // TMA destinations: 1024-byte aligned pieces when swizzled (tensor-core
    // path), 128-byte aligned rows otherwise.
    const bool tc = sc->R >= 4;
    const int w = sc->d % 64 == 0 ? 64 : (sc->d % 32 == 0 ? 32 : 16);
    const long long piece = (tc ? (long long)box_rows * w * 2 : (long long)box_rows * sc->d * 2) * sc->hp;
    if (piece % (tc ? 1024 : 128) != 0) return LA_ERR_UNSUPPORTED;
  }
  if (sc == nullptr || q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      cu_seqlens_k_dev == nullptr)
    return LA_ERR_INVALID;
  if (dt != LA_F16 && dt != LA_BF16) return LA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens_k_dev, 4))
    return LA_ERR_INVALID;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return LA_ERR_INVALID;
  if (workspace == nullptr || !aligned(workspace, 256)) return LA_ERR_WORKSPACE;
  la_schedule* s = const_cast<la_schedule*>(sc);
  if (s->kind == 0) {
    // Host CTAs wait for later CTAs inside the launch: all G must be resident at once.
    int sms = 0, per_sm = 0;
    la_status e = device_sms(&sms);
    if (e != LA_OK) return e;
    e = capacity(s->d, s->T, s->R, &per_sm, s->hp);
    if (e != LA_OK) return e;
    if ((int64_t)s->G > (int64_t)sms * per_sm) return LA_ERR_INVALID;
  }
  la_status e = ensure_uploaded(s);
  if (e != LA_OK) return e;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  la::KParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.cu = cu_seqlens_k_dev;
  p.sched_cu = s->dev + s->off_cu;
  p.cta_seg = s->dev + s->off_cta_seg;
  p.segs = s->dev + s->off_segs;
  p.out = out;
  const la::WsLayout wl = la::workspace_layout(s->G, s->d, s->R * s->hp);
  p.hdr = reinterpret_cast<uint32_t*>(ws);
  p.flags = reinterpret_cast<uint32_t*>(ws + wl.flags);
  p.recs = reinterpret_cast<float*>(ws + wl.recs);
  p.kv_rows = (long long)s->hkv * s->cu[s->batch];
  p.G = s->G;
  p.batch = s->batch;
  p.hq = s->hq;
  p.hkv = s->unit_heads();
  p.kv_heads = s->hkv;
  p.qscale = scale * 1.4426950408889634f;  // log2(e): scores in base-2 units
  p.spin_ns = s->spin_ns;
  p.skip_signal = s->skip_signal;
  p.trace = s->trace;
  p.out_dtype = out_dtype;
  p.kv_layout = kv_layout;
  if (kv_layout != la::kKvSlab) {
    p.kv_rows = kv_rows;
    p.box_rows = box_rows;
    p.page_size = page_size;
    p.bt_stride = bt_stride;
    p.block_table = kv->block_table;
  }
  cudaStream_t st = (cudaStream_t)stream;
  const int dtype = dt == LA_BF16 ? 1 : 0;
  p.grp = s->unit_grp();
  p.nq = s->nq;
  p.rows = s->unit_grp() * s->nq;
  p.stages = s->stages > 0 ? s->stages
                           : (s->kind == 0 && s->R <= 16 ? la::stream_stages(s->d, s->T, s->hp, kv_layout) : 0);
  p.shared_pieces = la::shared_merge_pieces(s->R * s->hp);
  cudaError_t ce = la::launch_decode(s->d, s->T, s->R, s->hp, dtype, p, st);
  if (ce != cudaSuccess) return LA_ERR_CUDA;
  if (s->kind == 1 && s->splits > 1) {
    la::CParams c;
    c.unit_host = s->dev + s->off_host;
    c.unit_fin = s->dev + s->off_fin;
    c.recs = p.recs;
    c.out = out;
    c.U = s->U;
    c.hq = s->hq;
    c.hkv = s->unit_heads();
    c.out_dtype = out_dtype;
    c.grp = s->unit_grp();
    c.nq = s->nq;
    c.rows = s->unit_grp() * s->nq;
    ce = la::launch_combine(s->d, s->R, c, st);
    if (ce != cudaSuccess) return LA_ERR_CUDA;
  }
  return LA_OK;
}

la_status la_decode_ex(const void* q, const void* k, const void* v, la_dtype dt, const int32_t* cu_seqlens_k_dev,
                       const la_schedule* s, void* workspace, void* out, la_dtype_out out_dt, float scale,
                       la_stream_t stream) {
  const la_kv_desc slab = {LA_KV_SLAB, nullptr, 0, 0, 0};
  return la_decode_kv(q, k, v, dt, cu_seqlens_k_dev, &slab, s, workspace, out, out_dt, scale, stream);
}

la_status la_decode(const void* q, const void* k, const void* v, la_dtype dt, const int32_t* cu_seqlens_k_dev,
                    const la_schedule* s, void* workspace, float* out, float scale, la_stream_t stream) {
  return la_decode_ex(q, k, v, dt, cu_seqlens_k_dev, s, workspace, out, LA_OUT_F32, scale, stream);
}

la_status la_decode_host(const void* q_host, const void* k_host, const void* v_host, la_dtype dt,
                         const int32_t* cu_seqlens_k_dev, const la_schedule* s, void* q_dev, void* k_dev,
                         void* v_dev, void* workspace, float* out_dev, float* out_host, float scale,
                         la_stream_t stream) {
  if (s == nullptr || q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr)
    return LA_ERR_INVALID;
  if (s->hp != 1) return LA_ERR_UNSUPPORTED;  // units of several kv heads read token-major or paged caches
  const size_t q_bytes = (size_t)s->batch * s->nq * s->hq * s->d * 2;
  const size_t kv_bytes = (size_t)s->hkv * (size_t)s->cu[s->batch] * s->d * 2;
  const size_t out_bytes = (size_t)s->batch * s->nq * s->hq * s->d * sizeof(float);
  // la_decode's own argument checks, made before any copy is enqueued
  if (q_dev == nullptr || k_dev == nullptr || v_dev == nullptr || out_dev == nullptr ||
      cu_seqlens_k_dev == nullptr)
    return LA_ERR_INVALID;
  if (dt != LA_F16 && dt != LA_BF16) return LA_ERR_INVALID;
  if (!aligned(q_dev, 16) || !aligned(k_dev, 16) || !aligned(v_dev, 16) || !aligned(out_dev, 16) ||
      !aligned(cu_seqlens_k_dev, 4))
    return LA_ERR_INVALID;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return LA_ERR_INVALID;
  if (workspace == nullptr || !aligned(workspace, 256)) return LA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(k_dev, k_host, kv_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(v_dev, v_host, kv_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return LA_ERR_CUDA;
  const la_status e = la_decode(q_dev, k_dev, v_dev, dt, cu_seqlens_k_dev, s, workspace, out_dev, scale, stream);
  if (e != LA_OK) return e;
  return cudaMemcpyAsync(out_host, out_dev, out_bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess ? LA_OK
                                                                                                   : LA_ERR_CUDA;
}

la_status la_get_status(void* workspace, la_stream_t stream) {
  if (workspace == nullptr) return LA_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LA_ERR_CUDA;
  uint32_t hdr[8] = {0};
  if (cudaMemcpy(hdr, workspace, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return LA_ERR_CUDA;
  const uint32_t code = hdr[la::kStatus];
  if (code != 0) {
    uint32_t zero[3] = {0, 0, 0};
    if (cudaMemcpy(static_cast<uint32_t*>(workspace) + la::kStatus, zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return LA_ERR_CUDA;
  }
  switch (code) {
    case 0: return LA_OK;
    case LA_ERR_INVALID: return LA_ERR_INVALID;
    case LA_ERR_TIMEOUT: return LA_ERR_TIMEOUT;
    default: return LA_ERR_CUDA;
  }
}

size_t la_schedule_export_size(const la_schedule* s) {
  if (s == nullptr) return 0;
  return 8 + (size_t)(s->G + 1) * 2 + (size_t)(s->U + 1) + s->segs.size() + (size_t)s->U * 2;
}

la_status la_schedule_export(const la_schedule* s, int32_t* buf, size_t n) {
  if (s == nullptr || buf == nullptr || n < la_schedule_export_size(s)) return LA_ERR_INVALID;
  size_t w = 0;
  const int32_t head[8] = {0x4C41, s->G, s->U, (int32_t)s->I, s->T,
                           (int32_t)(s->segs.size() / la::kSegWords), s->kind, s->splits};
  for (int32_t x : head) buf[w++] = x;
  for (int32_t x : s->cta_iter) buf[w++] = x;
  for (int32_t x : s->unit_iter) buf[w++] = x;
  for (int32_t x : s->cta_seg) buf[w++] = x;
  for (int32_t x : s->segs) buf[w++] = x;
  for (int32_t x : s->unit_host) buf[w++] = x;
  for (int32_t x : s->unit_fin) buf[w++] = x;
  return LA_OK;
}

la_status la_schedule_set_debug(la_schedule* s, int skip_signal_cta, long long spin_timeout_ns) {
  if (s == nullptr || spin_timeout_ns <= 0) return LA_ERR_INVALID;
  s->skip_signal = skip_signal_cta;
  s->spin_ns = spin_timeout_ns;
  return LA_OK;
}

la_status la_schedule_set_stages(la_schedule* s, int stages) {
  if (s == nullptr || stages < 0 || stages > 4 || stages == 1) return LA_ERR_INVALID;
  s->stages = stages;
  return LA_OK;
}

la_status la_schedule_set_trace(la_schedule* s, void* trace_dev) {
  if (s == nullptr) return LA_ERR_INVALID;
  if (trace_dev != nullptr && (reinterpret_cast<uintptr_t>(trace_dev) % 8) != 0) return LA_ERR_INVALID;
  s->trace = static_cast<unsigned long long*>(trace_dev);
  return LA_OK;
}

la_status la_device_capacity(int d, int grp, int* ctas_per_sm, int* num_sms) {
  if (ctas_per_sm == nullptr || num_sms == nullptr) return LA_ERR_INVALID;
  if (la::default_tile(d) == 0) return LA_ERR_UNSUPPORTED;
  const int rows = unit_rows(grp, 1, d);
  if (rows == 0) return LA_ERR_UNSUPPORTED;
  la_status e = device_sms(num_sms);
  if (e != LA_OK) return e;
  return capacity(d, rows > 16 ? la::wide_tile(d) : la::default_tile(d), instance_rows(rows), ctas_per_sm);
}

void la_schedule_destroy(la_schedule* s) {
  if (s == nullptr) return;
  if (s->dev != nullptr) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != s->device) cudaSetDevice(s->device);
    cudaFree(s->dev);
    if (cur >= 0 && cur != s->device) cudaSetDevice(cur);
  }
  delete s;
}

const char* la_status_string(la_status st) {
  switch (st) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID: return "invalid argument";
    case LA_ERR_UNSUPPORTED: return "unsupported shape";
    case LA_ERR_CUDA: return "CUDA error";
    case LA_ERR_TIMEOUT: return "a bounded wait inside the kernel ran out";
    case LA_ERR_WORKSPACE: return "bad workspace";
    default: return "unknown status";
  }
}

}  // extern "C"
