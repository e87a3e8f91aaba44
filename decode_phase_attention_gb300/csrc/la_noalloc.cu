// la_noalloc.cu -- la_decode_static: the decode call for callers that
// cannot allocate device memory.
//
// The kernel needs scratch beyond its inputs and outputs: the ready flags,
// the partial records of split units and the schedule's tables. la_decode
// takes that scratch as a caller-allocated workspace and uploads the tables
// into memory it allocates itself. This entry point instead keeps all of it
// in one fixed array of device memory compiled into the library, so it never
// calls cudaMalloc or cudaFree.
#include <cuda_runtime.h>

#include <mutex>

#include "la_internal.h"
#include "la_schedule.h"
#include "lean_attn.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB per GPU, held until exit

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// In host code g_static_scratch only names the symbol; its device address
// comes from cudaGetSymbolAddress, once per device, with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Which schedule's tables each device's array holds (its address and serial
// number; serial 0: none yet), so that a run of calls with one schedule
// copies the tables once instead of on every call.
struct Held {
  const la_schedule* s = nullptr;
  uint64_t serial = 0;
};
Held g_held[kMaxDevices];

la_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return LA_OK;
}

struct Layout {
  la::WsLayout ws;
  size_t cu, cta_seg, segs, host, fin, total;
};

// shared: two record slots per CTA where the instance can merge split units
// shared (la::record_slots); false: one, every unit merged at its host.
Layout layout_of(const la_schedule* s, bool shared) {
  Layout L;
  L.ws = la::workspace_layout(s->G, s->d, s->R * s->hp, shared);  // header, flags and records as in a workspace
  size_t off = la::align_up(L.ws.end, 256);
  auto table = [&off](size_t words) {
    const size_t at = off;
    off = la::align_up(off + words * sizeof(int32_t), 16);
    return at;
  };
  L.cu = table(s->cu.size());
  L.cta_seg = table(s->cta_seg.size());
  L.segs = table(s->dev_segs.size());
  L.host = table(s->unit_host.size());
  L.fin = table(s->unit_fin.size());
  L.total = off;
  return L;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaError_t put(unsigned char* base, size_t at, const std::vector<int32_t>& v, cudaStream_t st) {
  if (v.empty()) return cudaSuccess;
  return cudaMemcpyAsync(base + at, v.data(), v.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
}

}  // namespace

extern "C" la_status la_decode_static(const void* q, const void* k, const void* v, la_dtype dt,
                                      const int32_t* cu_seqlens_k_dev, const la_schedule* sc, float* out,
                                      float scale, la_stream_t stream) {
  if (sc == nullptr || q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      cu_seqlens_k_dev == nullptr)
    return LA_ERR_INVALID;
  if (dt != LA_F16 && dt != LA_BF16) return LA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens_k_dev, 4))
    return LA_ERR_INVALID;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return LA_ERR_INVALID;
  const la_schedule* s = sc;
  if (s->hp != 1) return LA_ERR_UNSUPPORTED;  // units of several kv heads read token-major or paged caches
  // Where the second record slot per CTA of a shared merge does not fit,
  // the 16-row kernel merges every split unit at its host (one slot).
  bool shared = true;
  Layout L = layout_of(s, true);
  if (L.total > kStaticScratchBytes && s->R < la::kWideInstanceRows) {
    L = layout_of(s, false);
    shared = false;
  }
  if (L.total > kStaticScratchBytes) return LA_ERR_WORKSPACE;  // schedule too large for the fixed array

  if (s->kind == 0) {  // host CTAs wait on later CTAs: all of the grid must be resident
    int per_sm = 0, sms = 0;
    la_status e = (la_status)la::device_sm_count(&sms);
    if (e != LA_OK) return e;
    e = (la_status)la::cached_capacity(s->d, s->T, s->R, s->hp, &per_sm);
    if (e != LA_OK) return e;
    if ((long long)s->G > (long long)per_sm * sms) return LA_ERR_INVALID;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
  void* addr = nullptr;
  const la_status e = scratch_address(dev, &addr);
  if (e != LA_OK) return e;
  unsigned char* base = static_cast<unsigned char*>(addr);
  cudaStream_t st = (cudaStream_t)stream;

  // The array keeps whatever the previous call left: clear the header
  // (epoch, done counter, status) and the ready flags; copy the tables
  // unless this device's array already holds this schedule's.
  if (cudaMemsetAsync(base, 0, L.ws.recs, st) != cudaSuccess) return LA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    Held& h = g_held[dev];
    if (h.s != s || h.serial != s->serial) {
      h = Held{};  // a failed copy leaves no schedule recorded
      if (put(base, L.cu, s->cu, st) != cudaSuccess || put(base, L.cta_seg, s->cta_seg, st) != cudaSuccess ||
          put(base, L.segs, s->dev_segs, st) != cudaSuccess || put(base, L.host, s->unit_host, st) != cudaSuccess ||
          put(base, L.fin, s->unit_fin, st) != cudaSuccess)
        return LA_ERR_CUDA;
      h.s = s;
      h.serial = s->serial;
    }
  }

  la::KParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.cu = cu_seqlens_k_dev;
  p.sched_cu = reinterpret_cast<const int32_t*>(base + L.cu);
  p.cta_seg = reinterpret_cast<const int32_t*>(base + L.cta_seg);
  p.segs = reinterpret_cast<const int32_t*>(base + L.segs);
  p.out = out;
  p.hdr = reinterpret_cast<uint32_t*>(base);
  p.flags = reinterpret_cast<uint32_t*>(base + L.ws.flags);
  p.recs = reinterpret_cast<float*>(base + L.ws.recs);
  p.kv_rows = (long long)s->hkv * s->cu[s->batch];
  p.G = s->G;
  p.batch = s->batch;
  p.hq = s->hq;
  p.hkv = s->unit_heads();
  p.kv_heads = s->hkv;
  p.qscale = scale * 1.4426950408889634f;
  p.spin_ns = s->spin_ns;
  p.skip_signal = s->skip_signal;
  p.trace = s->trace;
  const int dtype = dt == LA_BF16 ? 1 : 0;
  p.grp = s->unit_grp();
  p.nq = s->nq;
  p.rows = s->unit_grp() * s->nq;
  p.stages = s->stages > 0 ? s->stages
                           : (s->kind == 0 && s->R <= 16 ? la::stream_stages(s->d, s->T, s->hp, la::kKvSlab) : 0);
  p.shared_pieces = shared ? la::shared_merge_pieces(s->R * s->hp) : 0;
  cudaError_t ce = la::launch_decode(s->d, s->T, s->R, 1, dtype, p, st);
  if (ce != cudaSuccess) return LA_ERR_CUDA;
  if (s->kind == 1 && s->splits > 1) {
    la::CParams c;
    c.unit_host = reinterpret_cast<const int32_t*>(base + L.host);
    c.unit_fin = reinterpret_cast<const int32_t*>(base + L.fin);
    c.recs = p.recs;
    c.out = out;
    c.U = s->U;
    c.hq = s->hq;
    c.hkv = s->unit_heads();
    c.grp = s->unit_grp();
    c.nq = s->nq;
    c.rows = s->unit_grp() * s->nq;
    ce = la::launch_combine(s->d, s->R, c, st);
    if (ce != cudaSuccess) return LA_ERR_CUDA;
  }
  return LA_OK;
}
