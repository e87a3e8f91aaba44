// la_kernel.cuh -- the stream-K LeanAttention decode kernel for sm_103a.
//
// One launch computes every output of a decode-attention call (xllm-io
// paper review of LeanAttention, "3.5 execution flow" and "4.4 single
// kernel fusion"). CTA g walks the segments the host planner gave it:
//   kWhole    a whole (request, kv head) unit: LeanTile loop, normalise, store
//   kNonHost  the leading piece of a unit hosted by a lower CTA: LeanTile
//             loop, write the partial (m, l, O) to the workspace, release a
//             ready flag
//   kHost     the trailing piece of a unit: LeanTile loop, then for every
//             later CTA of the unit wait on its flag and merge its partial
//             with the rescaling reduction f ("3.2", part 2), normalise, store
//   kPartial  fixed-split baseline piece: write the partial, no flag
//
// Warp roles (288 threads, one CTA per SM):
//   warp 8:         producer. Streams the K and V rows of each LeanTile of
//                   every segment, in order, from HBM into a shared-memory
//                   ring of 2-4 stages (completion counted in bytes on one
//                   mbarrier per stage); lane 0 issues the slab copies, lane
//                   i the i-th page piece of a tile of a token-major or paged
//                   cache.
//   warps 0-7:      consumers. Each takes T/8 consecutive tokens of the tile
//                   and keeps online-softmax statistics m, l and the
//                   unnormalised output in fp32 ("3.3 LeanTile": S_f = Q K^T,
//                   update m and l, O_acc = P V + diag(rescale) O_acc).
// Two tile paths:
//   CUDA cores (query-head group 1 or 2, about 1-2 flop per K/V byte): a
//     tile's K rows (and V rows) are one contiguous run of the [hkv, L, d]
//     slab, moved by a 1-D bulk copy (cp.async.bulk). d/8 lanes share one
//     token (16 bytes each, whole rows per warp, no bank conflicts); q.k is
//     reduced across them with shuffles, P.V accumulates in registers.
//   tensor cores (4-16 query rows per kv head, up to 16 flop per byte, which
//     would saturate the fp32 pipes): tiles arrive by 2-D TMA
//     (cp.async.bulk.tensor) with 128-byte swizzle, so ldmatrix reads are
//     conflict-free. With the query rows as the N = 8 side of an m16n8k16
//     MMA (two blocks of 8 above 8 rows), S = K q^T
//     (tokens x heads) and O^T = V^T P (dims x heads) need no padding rows;
//     P moves from the accumulator layout to the operand layout with
//     movmatrix, and is split into a bf16/fp16 high and low part so that
//     the P.V product keeps fp32-level accuracy.
// At the end of a segment the lanes of a warp and then the 8 warps merge
// with f (the warps through shared memory); a host CTA then merges the
// partials of the unit's later CTAs (staged in the idle ring when there
// are many of them).
//
// Units of HP > 1 kv heads (token-major and paged caches with short rows):
// a tile holds T tokens of each of the unit's HP heads, loaded as the cache
// stores them (tile row = token * HP + head, so each load reads HP * d
// contiguous elements per token); the warps split into HP groups of NCW / HP,
// one group per head, and merge within their group.
//
// Scores are kept in base-2 units: scale*log2(e) multiplies q.k so that
// exp(s - m) becomes ex2(s2 - m2); m in the workspace records is in the
// same units (the records are internal to this kernel).
//
// Every wait is bounded (globaltimer). A wait that runs out records
// LA_ERR_TIMEOUT in the workspace header, raises a CTA-wide abort flag that
// makes every other wait return at once, the producer waits (bounded) for
// its copies still in flight, and the affected outputs are written as NaN.
//
// The kernel is launched as a programmatic dependent of the kernel before
// it on the stream and waits for that grid before touching memory
// (grid_dependency_sync), so back-to-back calls overlap only their launch.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "la_internal.h"

namespace la {

constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kStatusInvalid = 1;  // LA_ERR_INVALID
constexpr uint32_t kStatusTimeout = 4;  // LA_ERR_TIMEOUT

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 1-D bulk copy global -> shared, completion signalled on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// 2-D tiled TMA load of box (x, y) of tensor map `tmap` into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// 3-D tiled TMA load of box (x, y, z) of tensor map `tmap` into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tmap, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
__device__ __forceinline__ float ex2(float x) {  // 2^x; ex2(-inf) = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ------------------------------------------------------------ element types
template <typename E>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  // bf16 is the upper half of an fp32: widening is a shift / mask.
  __device__ static __forceinline__ void to_f32(const uint4& x, float f[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  // Pack (lo, hi) into a bf16x2 register, round to nearest even.
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ float2 unpack(uint32_t x) {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
  }
  __device__ static __forceinline__ void mma(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static constexpr bool kBf16 = true;
};
template <>
struct Elem<__half> {
  __device__ static __forceinline__ void to_f32(const uint4& x, float f[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ float2 unpack(uint32_t x) {
    return __half22float2(*reinterpret_cast<const __half2*>(&x));
  }
  __device__ static __forceinline__ void mma(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  static constexpr bool kBf16 = false;
};

// ------------------------------------------------------------ configuration
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int T_, int GRP, int HP = 1>
struct Cfg {
  static constexpr int DIM = D;                     // head dim
  static constexpr int HPU = HP;                    // kv heads per unit
  static constexpr int T = T_;                      // LeanTile tokens (of each kv head of the unit)
  static constexpr int ROWS = T * HP;               // K (and V) rows of a tile: T tokens x HP kv heads
  static constexpr bool TC = (GRP >= 4);            // tensor-core tile path
  // consumer warps: 8, or fewer when an MMA tile of 16 tokens per warp needs it
  static constexpr int NCW = TC ? cmin(8, ROWS / 16) : 8;
  static constexpr int NCT = NCW * 32;              // consumer threads
  static constexpr int NTHREADS = NCT + 32;         // + producer warp
  static constexpr int WPH = NCW / HP;              // consumer warps per kv head of the unit
  static constexpr int TPW = T / WPH;               // tokens per warp per tile
  // CUDA-core path: d/8 active lanes per token (16 bytes each), rounded up
  // to a power-of-two lane group; the spare lanes of a group idle.
  static constexpr int ACT = D / 8;
  static constexpr int LPT = ACT <= 8 ? 8 : (ACT <= 16 ? 16 : 32);
  static constexpr int TPS = 32 / LPT;              // tokens per warp step
  static constexpr int STEPS = TPW / TPS;
  static constexpr int CH = (GRP <= 2) ? cmin(STEPS, 8) : (GRP == 4 ? cmin(STEPS, 4) : cmin(STEPS, 2));
  // tensor-core path: TMA boxes of W columns (W*2-byte rows, swizzled)
  static constexpr int W = (D % 64 == 0) ? 64 : ((D % 32 == 0) ? 32 : 16);
  static constexpr int RB = W * 2;                  // box row bytes: 128, 64 or 32
  static constexpr int NB = D / W;                  // boxes per tile per tensor
  static constexpr int MT = TPW / 16;               // 16-token MMA tiles per warp
  static constexpr int KS = D / 16;                 // 16-wide steps over the head dim
  static constexpr int NB8 = (GRP + 7) / 8;         // 8-row blocks of the tensor-core path
  static constexpr int TILE_ELEMS = ROWS * D;
  static constexpr int STAGE_BYTES = 2 * TILE_ELEMS * 2;
  static constexpr int REC = D + kRecO;             // [m, l, 0, 0, O[d]]
  static constexpr int RS = record_stride(D, HP * GRP);  // floats per CTA record in the workspace
  static constexpr size_t MERGE_BYTES = (size_t)NCW * GRP * REC * 4;
  // shared memory for a ring of 2-4 stages within 192 KiB (less when a large
  // merge area leaves less room); a launch may use fewer of them
  // (KParams::stages)
  static constexpr int RING_ROOM = cmin(196608, 232448 - (int)MERGE_BYTES - (2 * 4 * 8 + 16) - 1024);
  static constexpr int STAGES = cmax(2, cmin(4, RING_ROOM / STAGE_BYTES));
  static constexpr size_t KV_BYTES = (size_t)STAGES * STAGE_BYTES;
  static constexpr size_t BAR_BYTES = 2 * STAGES * 8 + 16 + 16;  // full, empty, 2 flag words, 2 staging barriers
  static constexpr size_t SMEM = KV_BYTES + MERGE_BYTES + BAR_BYTES + 1024;  // + alignment slack
  static constexpr int V4 = (HP * GRP * D / 4 + NCT - 1) / NCT;  // vectors of 4 (row, dim) outputs per consumer thread
  static constexpr int PB = cmax(1, cmin(4, 4 / V4));  // peer records per batch of host-merge loads
  // Host merge of many peers, in the idle ring and merge area (contiguous):
  // two buffers of up to NBAT staged peer records, then per-row scalars
  // (running maximum, running l, this batch's rescale, NBAT peer weights).
  static constexpr int MROWS = HP * GRP;            // record rows
  static constexpr int NBAT_MAX = 64;
  static constexpr size_t SCAL_BYTES = ((size_t)MROWS * (3 + NBAT_MAX) * 4 + 15) / 16 * 16;
  static constexpr int NBAT = cmin(NBAT_MAX, (int)((KV_BYTES + MERGE_BYTES - SCAL_BYTES) / (2 * RS * 4)));
  static constexpr size_t SCAL_OFF = (size_t)2 * NBAT * RS * 4;
  static_assert(D % 16 == 0 && T % 16 == 0, "tile shape");
  static_assert((HP == 1 || HP == 2 || HP == 4 || HP == 8) && NCW % HP == 0 && T % WPH == 0, "kv heads per unit");
  static_assert(STEPS % CH == 0 && TPW % TPS == 0, "CUDA-core tile shape");
  static_assert(!TC || (TPW % 16 == 0 && (GRP <= 8 || GRP % 8 == 0) && GRP <= 16), "tensor-core tile shape");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(NBAT >= 1 && SCAL_OFF + SCAL_BYTES <= KV_BYTES + MERGE_BYTES, "host-merge staging");
};

// a * x + y and a * x on 4-vectors.
__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 scale4(float a, float4 x) { return make_float4(a * x.x, a * x.y, a * x.z, a * x.w); }

// Output element store (fp32, fp16 or bf16, chosen per call).
__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_dtype) {
  if (out_dtype == 0)
    static_cast<float*>(out)[idx] = v;
  else if (out_dtype == 1)
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}
// Two consecutive outputs (idx even) as fp32, fp16 or bf16.
__device__ __forceinline__ void store_out2(void* out, size_t idx, float a, float b, int out_dtype) {
  if (out_dtype == 0) {
    *reinterpret_cast<float2*>(static_cast<float*>(out) + idx) = make_float2(a, b);
  } else if (out_dtype == 1) {
    __half2 x = __floats2half2_rn(a, b);
    *reinterpret_cast<uint32_t*>(static_cast<__half*>(out) + idx) = *reinterpret_cast<uint32_t*>(&x);
  } else {
    __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
    *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(out) + idx) = *reinterpret_cast<uint32_t*>(&x);
  }
}
// Four consecutive outputs (idx a multiple of 4) as fp32, fp16 or bf16.
__device__ __forceinline__ void store_out4(void* out, size_t idx, float a, float b, float c, float d,
                                           int out_dtype) {
  if (out_dtype == 0) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + idx) = make_float4(a, b, c, d);
  } else if (out_dtype == 1) {
    __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, d);
    *reinterpret_cast<uint2*>(static_cast<__half*>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t*>(&x), *reinterpret_cast<uint32_t*>(&y));
  } else {
    __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, d);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + idx) =
        make_uint2(*reinterpret_cast<uint32_t*>(&x), *reinterpret_cast<uint32_t*>(&y));
  }
}

// Element offset / D of query row r of unit (b, kvh) in q and out
// ([batch, nq, hq, d]): query token r / grp, head kvh * grp + r % grp (kvh
// and grp count unit heads: a query block of a kv head is a head of its own).
template <typename P>
__device__ __forceinline__ size_t row_index(const P& p, int b, int kvh, int r) {
  return ((size_t)b * p.nq + r / p.grp) * p.hq + (size_t)kvh * p.grp + r % p.grp;
}

// Tokens of tile t (0-based inside the request) that row r may attend to:
// query token i of nq sits at position L - nq + i and sees keys up to it.
__device__ __forceinline__ int row_visible(const KParams& p, long long L, int t, int T, int r) {
  const long long lim = L - (p.nq - 1 - r / p.grp) - (long long)t * T;
  return lim < 0 ? 0 : (lim > T ? T : (int)lim);
}

// Record the first error of the launch in the workspace header.
__device__ __forceinline__ void record_error(uint32_t* hdr, uint32_t code, int cta, int peer) {
  if (atomicCAS(&hdr[kStatus], 0u, code) == 0u) {
    hdr[kInfoCta] = (uint32_t)cta;
    hdr[kInfoPeer] = (uint32_t)peer;
  }
}

// Bounded wait on an mbarrier phase. Returns false if the abort flag is up
// or the limit ran out (the caller records the error).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if ((long long)(global_ns() - t0) > limit_ns) return false;
    }
  }
}

// The schedule was planned with host offsets; the kernel reads the device
// copy the caller passes. They must agree before any address is formed.
__device__ __forceinline__ bool unit_offsets_ok(const KParams& p, int b) {
  return p.cu[b] == p.sched_cu[b] && p.cu[b + 1] == p.sched_cu[b + 1];
}

// Stages of the ring this launch cycles through: the host's choice
// (KParams::stages) within [2, STAGES]; 0 (or out of range) means STAGES.
template <class C>
__device__ __forceinline__ int ring_stages(const KParams& p) {
  return (p.stages >= 2 && p.stages < C::STAGES) ? p.stages : C::STAGES;
}

// ------------------------------------------------------------------ producer
// C: the kernel's configuration (tile tokens T, head dim DIM, kv heads per
// unit HPU, tensor-core boxes TC / W / NB, TILE_ELEMS and STAGES).
template <class C, typename E>
__device__ __forceinline__ void produce(const KParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv, int g,
                                        E* kv, uint64_t* full, uint64_t* empty, volatile int* abort_flag) {
  // Run by the whole producer warp. Lane 0 posts byte counts and issues the
  // slab-layout copies; for token-major and paged caches lane i issues the
  // load of the i-th piece of a tile (a tile spans up to T / 16 pages), so
  // small pages do not serialise on one thread. A unit of HP > 1 kv heads
  // (token-major and paged caches only) loads the HP heads of each token
  // row together: HP * d contiguous elements per row, kept interleaved in
  // shared memory (tile row = token * HP + head).
  constexpr int D = C::DIM, HP = C::HPU;
  const int lane = threadIdx.x & 31;
  const bool leader = lane == 0;
  const uint64_t pol = l2_evict_first_policy();
  const bool tma3 = p.kv_layout != kKvSlab;
  if (leader && (C::TC || tma3)) {
    prefetch_tmap(tmk);
    prefetch_tmap(tmv);
  }
  const int s_begin = p.cta_seg[g], s_end = p.cta_seg[g + 1];
  const int ns = ring_stages<C>(p);
  int stage = 0;
  uint32_t phase = 1;  // a fresh barrier counts its previous (odd) phase as complete
  long long issued = 0;
  bool aborted = false;
  for (int si = s_begin; si < s_end && !aborted; ++si) {
    // the schedule's own offsets: every copy stays inside the K/V extent the
    // schedule was planned for, whatever the caller's device offsets hold
    const int4 w0 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords);
    const int4 w1 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords + 4);
    const int4 w2 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords + 8);
    const int t0 = w0.y, t1 = w0.z;
    const long long L = w1.y;
    const long long row0 = (long long)(((unsigned long long)(unsigned)w1.w << 32) | (unsigned)w1.z);
    const int cu_b = w2.x, b = w2.y, kvh = w2.z;
    for (int t = t0; t < t1; ++t) {
      const long long rem = L - (long long)t * C::T;
      const int ntok = rem < C::T ? (int)rem : C::T;
      const int br = tma3 ? p.box_rows : C::T;
      const int nload = (ntok + br - 1) / br;  // pieces that start inside the context
      // this lane's piece: its first token row in the cache (read before the
      // wait, so a page id's latency overlaps it)
      int row = 0;
      if (tma3 && lane < nload) {
        const int tok = t * C::T + lane * br;
        if (p.kv_layout == kKvTokenMajor) {
          row = cu_b + tok;
        } else {
          const int page = p.block_table[(size_t)b * p.bt_stride + tok / p.page_size];
          row = page * p.page_size + tok % p.page_size;
        }
      }
      bool free_slot = mbar_wait_bounded(&empty[stage], phase, abort_flag, p.spin_ns);
      free_slot = __all_sync(kFull, free_slot);
      if (!free_slot) {
        if (leader) {
          record_error(p.hdr, kStatusTimeout, g, -1);
          *abort_flag = 1;
        }
        aborted = true;
        break;
      }
      E* ks = kv + (size_t)stage * 2 * C::TILE_ELEMS;
      if (tma3) {
        // Token-major or paged cache, seen as [rows, hkv, d]: box_rows token
        // rows of the unit's HP kv heads per load; the consumers mask the
        // tail tokens.
        if (leader) mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * nload * br * HP * D * 2));
        __syncwarp();
        if (lane < nload) {
          if (C::TC) {
#pragma unroll
            for (int bk = 0; bk < C::NB; ++bk) {
              const int off = bk * C::ROWS * C::W + lane * br * HP * C::W;
              tma_load_3d(ks + off, tmk, bk * C::W, kvh, row, &full[stage], pol);
              tma_load_3d(ks + C::TILE_ELEMS + off, tmv, bk * C::W, kvh, row, &full[stage], pol);
            }
          } else {
            tma_load_3d(ks + lane * br * HP * D, tmk, 0, kvh, row, &full[stage], pol);
            tma_load_3d(ks + C::TILE_ELEMS + lane * br * HP * D, tmv, 0, kvh, row, &full[stage], pol);
          }
        }
      } else if (HP == 1 && leader) {  // slab layout: the host accepts only HP = 1
        if (C::TC) {
          // Whole boxes of T rows: rows past the slab are the next slab's (or
          // zero fill past the tensor) and are masked by the consumers.
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(2 * C::TILE_ELEMS * 2));
          const int y = (int)(row0 + (long long)t * C::T);
#pragma unroll
          for (int bk = 0; bk < C::NB; ++bk) {
            tma_load_2d(ks + bk * C::T * C::W, tmk, bk * C::W, y, &full[stage], pol);
            tma_load_2d(ks + C::TILE_ELEMS + bk * C::T * C::W, tmv, bk * C::W, y, &full[stage], pol);
          }
        } else {
          const uint32_t bytes = (uint32_t)ntok * D * 2u;
          mbar_arrive_expect_tx(&full[stage], 2u * bytes);
          const E* src_k = static_cast<const E*>(p.k) + (row0 + (long long)t * C::T) * D;
          const E* src_v = static_cast<const E*>(p.v) + (row0 + (long long)t * C::T) * D;
          bulk_g2s(ks, src_k, bytes, &full[stage], pol);
          bulk_g2s(ks + C::TILE_ELEMS, src_v, bytes, &full[stage], pol);
        }
      }
      ++issued;
      if (++stage == ns) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (aborted && leader) {
    // Do not leave the CTA while copies into its shared memory are in flight:
    // wait (bounded) for the latest fill of every stage that was used.
    for (int s = 0; s < ns; ++s) {
      const long long fills = issued / ns + (s < issued % ns ? 1 : 0);
      if (fills == 0) continue;
      const uint32_t parity = (uint32_t)((fills - 1) & 1);
      volatile int no_abort = 0;
      mbar_wait_bounded(&full[s], parity, &no_abort, p.spin_ns);
    }
  }
  __syncwarp();
}

// Wait for the next stage; false (for the whole warp) if it never came.
template <int D, int T, int GRP>
__device__ __forceinline__ bool wait_tile(const KParams& p, int g, uint64_t* full, int stage, uint32_t phase,
                                          volatile int* abort_flag, int lane) {
  bool have = mbar_wait_bounded(&full[stage], phase, abort_flag, p.spin_ns);
  have = __all_sync(kFull, have);
  if (!have && lane == 0) {
    if (!*abort_flag) record_error(p.hdr, kStatusTimeout, g, -1);
    *abort_flag = 1;
  }
  if (p.trace != nullptr && threadIdx.x == 0) {
    unsigned long long* tr = p.trace + (size_t)g * kTraceWords;
    if (tr[kTrFirstTile] == 0ull) tr[kTrFirstTile] = global_ns();
    tr[kTrTiles] += 1ull;
  }
  return have;
}

// ----------------------------------------------- CUDA-core tile path (grp 1, 2)
// Runs the segment's tiles and leaves this warp's (m, l, O) for every head
// of the group in its slot of the merge area.
template <int D, int T, int GRP, typename E, int HP>
__device__ __forceinline__ void warp_segment_cc(const KParams& p, int g, int b, int kvh0, long long L, int t0,
                                                int n_tiles, bool ok, const E* kv, uint64_t* full, uint64_t* empty,
                                                int& stage, uint32_t& phase, volatile int* abort_flag,
                                                float* wrec) {
  using C = Cfg<D, T, GRP, HP>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hh = HP == 1 ? 0 : warp / C::WPH;  // kv head of the unit this warp works on
  const int kvh = kvh0 + hh;
  const int gl = lane % C::LPT;   // which 8-element chunk of the row
  const int ts = lane / C::LPT;   // which token of the warp step
  const bool act = gl < C::ACT;   // spare lanes of a group (d = 80, 96) idle
  const int c0 = act ? gl * 8 : 0;
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

  float qf[GRP][8];
#pragma unroll
  for (int j = 0; j < GRP; ++j) {
    const uint4 raw =
        act ? *reinterpret_cast<const uint4*>(static_cast<const E*>(p.q) + row_index(p, b, kvh, j) * D + c0)
            : zero4;
    Elem<E>::to_f32(raw, qf[j]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[j][e] *= p.qscale;
  }
  float m[GRP], l[GRP], o[GRP][8];
#pragma unroll
  for (int j = 0; j < GRP; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[j][e] = 0.f;
  }

  for (int it = 0; it < n_tiles; ++it) {
    const long long rem = L - (long long)(t0 + it) * C::T;
    const int ntok = rem < C::T ? (int)rem : C::T;
    int vis[GRP];  // tokens of this tile each row may attend to
#pragma unroll
    for (int j = 0; j < GRP; ++j) vis[j] = row_visible(p, L, t0 + it, C::T, j);
    if (wait_tile<D, T, GRP>(p, g, full, stage, phase, abort_flag, lane) && ok) {
      const E* Ks = kv + (size_t)stage * 2 * C::TILE_ELEMS;
      const E* Vs = Ks + C::TILE_ELEMS;
      const int wtok = (HP == 1 ? warp : warp % C::WPH) * C::TPW;
#pragma unroll
      for (int c = 0; c < C::STEPS; c += C::CH) {
        float s[C::CH][GRP];
#pragma unroll
        for (int st = 0; st < C::CH; ++st) {
          const int tok = wtok + (c + st) * C::TPS + ts;
          const uint4 raw = act ? *reinterpret_cast<const uint4*>(Ks + (tok * HP + hh) * D + c0) : zero4;
          float kf[8];
          Elem<E>::to_f32(raw, kf);
#pragma unroll
          for (int j = 0; j < GRP; ++j) {
            float a0 = qf[j][0] * kf[0], a1 = qf[j][1] * kf[1];
#pragma unroll
            for (int e = 2; e < 8; e += 2) {
              a0 = fmaf(qf[j][e], kf[e], a0);
              a1 = fmaf(qf[j][e + 1], kf[e + 1], a1);
            }
            s[st][j] = a0 + a1;
          }
        }
#pragma unroll
        for (int st = 0; st < C::CH; ++st)
#pragma unroll
          for (int j = 0; j < GRP; ++j)
#pragma unroll
            for (int off = C::LPT / 2; off >= 1; off >>= 1) s[st][j] += __shfl_xor_sync(kFull, s[st][j], off);
#pragma unroll
        for (int st = 0; st < C::CH; ++st) {
          const int tok = wtok + (c + st) * C::TPS + ts;
#pragma unroll
          for (int j = 0; j < GRP; ++j)
            if (tok >= vis[j]) s[st][j] = -INFINITY;
        }
        // online softmax: new max, rescale, exponentiate
#pragma unroll
        for (int j = 0; j < GRP; ++j) {
          float mx = s[0][j];
#pragma unroll
          for (int st = 1; st < C::CH; ++st) mx = fmaxf(mx, s[st][j]);
          const float mn = fmaxf(m[j], mx);
          if (mn == -INFINITY) {
#pragma unroll
            for (int st = 0; st < C::CH; ++st) s[st][j] = 0.f;
            continue;
          }
          const float alpha = ex2(m[j] - mn);
          m[j] = mn;
          l[j] *= alpha;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[j][e] *= alpha;
#pragma unroll
          for (int st = 0; st < C::CH; ++st) {
            const float pj = ex2(s[st][j] - mn);
            s[st][j] = pj;
            l[j] += pj;
          }
        }
        // P.V
#pragma unroll
        for (int st = 0; st < C::CH; ++st) {
          const int tok = wtok + (c + st) * C::TPS + ts;
          if (tok < ntok && act) {
            const uint4 raw = *reinterpret_cast<const uint4*>(Vs + (tok * HP + hh) * D + c0);
            float vf[8];
            Elem<E>::to_f32(raw, vf);
#pragma unroll
            for (int j = 0; j < GRP; ++j)
#pragma unroll
              for (int e = 0; e < 8; ++e) o[j][e] = fmaf(s[st][j], vf[e], o[j][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == ring_stages<C>(p)) {
      stage = 0;
      phase ^= 1u;
    }
  }

  // merge the token slots of the warp (lanes with equal gl) with f
#pragma unroll
  for (int off = C::LPT; off < 32; off <<= 1) {
#pragma unroll
    for (int j = 0; j < GRP; ++j) {
      const float mo = __shfl_xor_sync(kFull, m[j], off);
      const float lo = __shfl_xor_sync(kFull, l[j], off);
      const float mn = fmaxf(m[j], mo);
      const float a = (m[j] == -INFINITY) ? 0.f : ex2(m[j] - mn);
      const float bw = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
      l[j] = a * l[j] + bw * lo;
      m[j] = mn;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float oo = __shfl_xor_sync(kFull, o[j][e], off);
        o[j][e] = a * o[j][e] + bw * oo;
      }
    }
  }
  if (ts == 0 && act) {
#pragma unroll
    for (int j = 0; j < GRP; ++j) {
      float* r = wrec + j * C::REC;
      if (gl == 0) {
        r[0] = m[j];
        r[1] = l[j];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) r[kRecO + c0 + e] = o[j][e];
    }
  }
}

// ----------------------------------- tensor-core tile path (4, 8 or 16 rows)
// Swizzled shared-memory address (128-byte swizzle: 16-byte chunk c of row r
// sits at chunk c ^ (r mod 8)) of row `row`, chunk `c` of 64-column block bk.
template <int D, int T, int GRP, int HP>
__device__ __forceinline__ uint32_t swz(uint32_t tile_base, int bk, int row, int c) {
  using C = Cfg<D, T, GRP, HP>;
  return tile_base + (uint32_t)(bk * C::ROWS * C::RB + row * C::RB +
                                ((c ^ ((row * C::RB >> 7) & (C::RB / 16 - 1))) << 4));
}

template <int D, int T, int GRP, typename E, int HP>
__device__ __forceinline__ void warp_segment_tc(const KParams& p, int g, int b, int kvh0, long long L, int t0,
                                                int n_tiles, bool ok, const E* kv, uint64_t* full, uint64_t* empty,
                                                int& stage, uint32_t& phase, volatile int* abort_flag,
                                                float* wrec) {
  using C = Cfg<D, T, GRP, HP>;
  constexpr int NB8 = C::NB8;  // blocks of 8 query rows: the N = 8 side of each MMA
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hh = HP == 1 ? 0 : warp / C::WPH;  // kv head of the unit this warp works on
  const int kvh = kvh0 + hh;
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // fragment column pair
  // B operand of S = K q^T per block of 8 rows: q^T (16 dims x 8 rows), raw
  // q bits; rows past the unit's are zero columns that are never written out.
  uint32_t qb[NB8][C::KS][2];
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    const int r = nb * 8 + gq;
    const bool live = r < p.rows;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(static_cast<const E*>(p.q) + row_index(p, b, kvh, live ? r : 0) * D);
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      qb[nb][ks][0] = live ? qrow[(ks * 16 + 2 * tq) / 2] : 0u;
      qb[nb][ks][1] = live ? qrow[(ks * 16 + 2 * tq + 8) / 2] : 0u;
    }
  }
  // State for rows nb*8 + 2tq and nb*8 + 2tq + 1 of every block: m (uniform
  // over the 8 row groups), the thread's share of l, and O^T fragments
  // (dims x rows).
  float m[NB8][2], l[NB8][2], o[NB8][C::KS][4];
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    m[nb][0] = m[nb][1] = -INFINITY;
    l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
    for (int dm = 0; dm < C::KS; ++dm)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[nb][dm][i] = 0.f;
  }

  const uint32_t kv_base = smem_u32(kv);
  for (int it = 0; it < n_tiles; ++it) {
    const long long rem = L - (long long)(t0 + it) * C::T;
    const int ntok = rem < C::T ? (int)rem : C::T;
    if (wait_tile<D, T, GRP>(p, g, full, stage, phase, abort_flag, lane) && ok) {
      const uint32_t kb = kv_base + (uint32_t)(stage * 2 * C::TILE_ELEMS * 2);
      const uint32_t vb = kb + (uint32_t)(C::TILE_ELEMS * 2);
      const int wtok = (HP == 1 ? warp : warp % C::WPH) * C::TPW;
      // S = K q^T for the warp's TPW tokens: MT tiles of 16 tokens x 8 rows
      // per block (one ldmatrix of K serves every block)
      float s[C::MT][NB8][4];
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) s[mt][nb][i] = 0.f;
        const int row = (wtok + mt * 16 + (lane & 15)) * HP + hh;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          uint32_t a[4];
          ldsm_x4(a, swz<D, T, GRP, HP>(kb, ks * 16 / C::W, row, (ks * 16 % C::W) / 8 + (lane >> 4)));
#pragma unroll
          for (int nb = 0; nb < NB8; ++nb) Elem<E>::mma(s[mt][nb], a, qb[nb][ks][0], qb[nb][ks][1]);
        }
      }
      // scale to base-2 units, mask tokens each row may not see, new maxima
      float mn[NB8][2], alpha[NB8][2];
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb) {
        const int vis0 = row_visible(p, L, t0 + it, C::T, nb * 8 + 2 * tq);
        const int vis1 = row_visible(p, L, t0 + it, C::T, nb * 8 + 2 * tq + 1);
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = wtok + mt * 16 + gq + ((i & 2) ? 8 : 0);
            s[mt][nb][i] = (tok < ((i & 1) ? vis1 : vis0)) ? s[mt][nb][i] * p.qscale : -INFINITY;
            mx[i & 1] = fmaxf(mx[i & 1], s[mt][nb][i]);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 4));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 8));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 16));
          mn[nb][h] = fmaxf(m[nb][h], mx[h]);
          alpha[nb][h] = (m[nb][h] == -INFINITY) ? 0.f : ex2(m[nb][h] - mn[nb][h]);
          if (mn[nb][h] == -INFINITY) alpha[nb][h] = 1.f;  // nothing seen yet
          m[nb][h] = mn[nb][h];
          l[nb][h] *= alpha[nb][h];
        }
#pragma unroll
        for (int dm = 0; dm < C::KS; ++dm) {
          o[nb][dm][0] *= alpha[nb][0];
          o[nb][dm][1] *= alpha[nb][1];
          o[nb][dm][2] *= alpha[nb][0];
          o[nb][dm][3] *= alpha[nb][1];
        }
      }
      // Rows past the context may hold anything (another request's tokens,
      // an unused page slot): their P is zero, but 0 * NaN is not, so the
      // warp clears its own V rows there before the P.V product.
      if (ntok < C::T && wtok + C::TPW > ntok) {
        constexpr int CHUNKS = C::RB / 16;  // 16-byte chunks per row and box
        for (int idx = lane; idx < C::TPW * C::NB * CHUNKS; idx += 32) {
          const int tok = wtok + idx / (C::NB * CHUNKS);
          const int rest = idx % (C::NB * CHUNKS);
          if (tok >= ntok) {
            const uint32_t a = vb + (uint32_t)((rest / CHUNKS) * C::ROWS * C::RB + (tok * HP + hh) * C::RB +
                                               (rest % CHUNKS) * 16);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
          }
        }
        __syncwarp();
      }
      // P = 2^(s - m), split into high and low 16-bit parts; O^T += V^T P
      // (one ldmatrix of V^T serves every block)
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
        uint32_t bh[NB8][2], bl[NB8][2];
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb) {
          float pv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float mi = mn[nb][i & 1];
            pv[i] = (mi == -INFINITY) ? 0.f : ex2(s[mt][nb][i] - mi);
            l[nb][i & 1] += pv[i];
          }
          const uint32_t h01 = Elem<E>::pack(pv[0], pv[1]);
          const uint32_t h23 = Elem<E>::pack(pv[2], pv[3]);
          const float2 f01 = Elem<E>::unpack(h01), f23 = Elem<E>::unpack(h23);
          const uint32_t l01 = Elem<E>::pack(pv[0] - f01.x, pv[1] - f01.y);
          const uint32_t l23 = Elem<E>::pack(pv[2] - f23.x, pv[3] - f23.y);
          bh[nb][0] = movmatrix_trans(h01);
          bh[nb][1] = movmatrix_trans(h23);
          bl[nb][0] = movmatrix_trans(l01);
          bl[nb][1] = movmatrix_trans(l23);
        }
        const int vrow = (wtok + mt * 16 + (lane & 7) + ((lane >> 4) << 3)) * HP + hh;
#pragma unroll
        for (int dm = 0; dm < C::KS; ++dm) {
          uint32_t a[4];
          ldsm_x4_trans(a, swz<D, T, GRP, HP>(vb, dm * 16 / C::W, vrow, (dm * 16 % C::W) / 8 + ((lane >> 3) & 1)));
#pragma unroll
          for (int nb = 0; nb < NB8; ++nb) {
            Elem<E>::mma(o[nb][dm], a, bh[nb][0], bh[nb][1]);
            Elem<E>::mma(o[nb][dm], a, bl[nb][0], bl[nb][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == ring_stages<C>(p)) {
      stage = 0;
      phase ^= 1u;
    }
  }

  // l: sum the shares of the 8 row groups (m is already common to them)
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l[nb][h] += __shfl_xor_sync(kFull, l[nb][h], 4);
      l[nb][h] += __shfl_xor_sync(kFull, l[nb][h], 8);
      l[nb][h] += __shfl_xor_sync(kFull, l[nb][h], 16);
    }
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int head = nb * 8 + 2 * tq + h;
      if (head < p.rows) {
        float* r = wrec + head * C::REC;
        if (gq == 0) {
          r[0] = m[nb][h];
          r[1] = l[nb][h];
        }
#pragma unroll
        for (int dm = 0; dm < C::KS; ++dm) {
          r[kRecO + dm * 16 + gq] = o[nb][dm][h];
          r[kRecO + dm * 16 + gq + 8] = o[nb][dm][2 + h];
        }
      }
    }
}

// ------------------------------------------------------------------ consumers
// The rescaling reduction f of one output element: (M, Ls, O) <- f((M, Ls, O),
// (m2, l2, o2)) in base-2 units; (-inf, 0, 0) is the identity and a NaN m2
// (a poisoned partial) propagates through its weight.
__device__ __forceinline__ void merge_f(float& M, float& Ls, float& O, float m2, float l2, float o2) {
  const float mn = fmaxf(M, m2);
  if (mn == -INFINITY) return;
  const float a = (M == -INFINITY) ? 0.f : ex2(M - mn);
  const float bw = (m2 == -INFINITY) ? 0.f : ex2(m2 - mn);
  Ls = a * Ls + bw * l2;
  O = a * O + bw * o2;
  M = mn;
}
// The same for 4 outputs of one row (one m and l).
__device__ __forceinline__ void merge_f4(float& M, float& Ls, float4& O, float m2, float l2, float4 o2) {
  const float mn = fmaxf(M, m2);
  if (mn == -INFINITY) return;
  const float a = (M == -INFINITY) ? 0.f : ex2(M - mn);
  const float bw = (m2 == -INFINITY) ? 0.f : ex2(m2 - mn);
  Ls = a * Ls + bw * l2;
  O = fma4(bw, o2, scale4(a, O));
  M = mn;
}

// The host merge of many peers on the CTA's last segment (called from
// consume). Out of line: compiled inline, its code slowed the CUDA-core tile
// loop of the d = 80 and 96 instances by 12 % (same-box A/B, one CTA per
// unit and stream-K), though the loop's own code did not change.
template <class C, typename E>
__device__ __noinline__ void host_merge_staged(const KParams& p, int g, int npeer, E* kv, uint64_t* stg, float* M,
                                               float* Lsum, float4* O, bool* fail) {
  constexpr int D = C::DIM;
  constexpr int kVecs = C::MROWS * D / 4;  // vectors of 4 consecutive outputs of a unit
  const int tid = threadIdx.x, warp = tid >> 5;
  // Many peers, and the CTA's last segment: every tile has been
  // consumed and the producer issues no more copies, so the ring
  // and the merge area after it (read above) are idle. The peers'
  // records come in by bulk copies (one per batch: the records of
  // consecutive CTAs are contiguous) in batches of up to NBAT into
  // two buffers, so the next batch's copy overlaps this batch's
  // merge. f is associative, so a batch of k partials reduces in
  // one step: per record row, the new maximum and the rescale of
  // the running partial, then every peer's weight 2^(m - max) --
  // each computed once per (row, peer) into shared memory -- then
  // the weighted sums of O (16-byte vectors) and of l.
  constexpr int kRows = C::MROWS;
  float* scal = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(kv) + C::SCAL_OFF);
  float* s_m = scal;              // [kRows] running maximum
  float* s_a = scal + kRows;      // [kRows] rescale of the running partial in this batch
  float* s_l = scal + 2 * kRows;  // [kRows] running l
  float* s_w = scal + 3 * kRows;  // [NBAT][kRows] peer weights of this batch
#pragma unroll
  for (int i = 0; i < C::V4; ++i) {
    const int v = tid + i * C::NCT;
    if (v < kVecs && 4 * v % D == 0) {
      s_m[4 * v / D] = M[i];
      s_l[4 * v / D] = Lsum[i];
    }
  }
  // A few KB (long MHA contexts: a handful of one-row records)
  // arrive sooner as every thread's 16-byte copies; more, as one
  // bulk copy per batch.
  const bool by_thread = (size_t)npeer * C::RS * 4 <= 32768;
  auto issue = [&](int first, int n, int buf) {
    unsigned char* dst = reinterpret_cast<unsigned char*>(kv) + (size_t)buf * C::NBAT * C::RS * 4;
    const float* src = p.recs + (size_t)(g + 1 + first) * C::RS;
    if (by_thread) {
      const uint32_t d0 = smem_u32(dst);
      for (int i = tid; i < n * (C::RS / 4); i += C::NCT)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d0 + 16u * (uint32_t)i),
                     "l"(src + 4 * (size_t)i)
                     : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    } else if (tid == 0) {
      const uint32_t bytes = (uint32_t)n * (uint32_t)(C::RS * 4);
      asm volatile("fence.proxy.async.global;" ::: "memory");  // records written by other CTAs
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the ring was last read here
      mbar_arrive_expect_tx(&stg[buf], bytes);
      bulk_g2s(dst, src, bytes, &stg[buf], l2_evict_first_policy());
    }
  };
  const int nbat = (npeer + C::NBAT - 1) / C::NBAT;
  issue(0, npeer < C::NBAT ? npeer : C::NBAT, 0);
  bool staged = true;
  for (int bi = 0; bi < nbat; ++bi) {
    const int first = bi * C::NBAT;
    const int n = npeer - first < C::NBAT ? npeer - first : C::NBAT;
    if (bi + 1 < nbat) {
      const int rest = npeer - first - C::NBAT;
      issue(first + C::NBAT, rest < C::NBAT ? rest : C::NBAT, (bi + 1) & 1);
    }
    if (by_thread) {
      if (bi + 1 < nbat)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      else
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
      // an issued copy is waited for (bounded) even after an abort
      volatile int no_abort = 0;
      if (!mbar_wait_bounded(&stg[bi & 1], (uint32_t)(bi >> 1) & 1u, &no_abort, p.spin_ns)) staged = false;
    }
    consumer_sync(C::NCT);  // batch bi is in shared memory (and s_m, s_l written)
    const float* st = reinterpret_cast<const float*>(kv) + (size_t)(bi & 1) * C::NBAT * C::RS;
    // per row, one warp (lanes over the batch's peers): the new
    // maximum, the rescale of the running partial, every peer's
    // weight and the new l
    static_assert(C::NBAT <= 64, "two peers per lane");
    for (int rr = warp; rr < kRows; rr += C::NCW) {
      const int lane = tid & 31;
      const float mo = s_m[rr];
      float mu[2], lu[2];
      float mb = mo;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = lane + 32 * q;
        mu[q] = u < n ? st[u * C::RS + rr * C::REC] : -INFINITY;
        lu[q] = u < n ? st[u * C::RS + rr * C::REC + 1] : 0.f;
        mb = fmaxf(mb, mu[q]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, off));
      float ls = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = lane + 32 * q;
        const float w = (mu[q] == -INFINITY) ? 0.f : ex2(mu[q] - mb);  // NaN m (poisoned) propagates
        if (u < n) s_w[u * kRows + rr] = w;
        ls = fmaf(w, lu[q], ls);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(kFull, ls, off);
      if (lane == 0) {
        const float a = (mb == -INFINITY || mo == -INFINITY) ? (mb == -INFINITY ? 1.f : 0.f) : ex2(mo - mb);
        s_a[rr] = a;
        s_m[rr] = mb;
        s_l[rr] = fmaf(a, s_l[rr], ls);
      }
    }
    consumer_sync(C::NCT);  // the batch's scalars are in shared memory
    // the weighted sums of O: peers outer, this thread's vectors
    // inner (V4 independent chains per step, 16-byte loads)
    {
      const float* rp[C::V4];
      const float* wp[C::V4];
#pragma unroll
      for (int i = 0; i < C::V4; ++i) {
        const int v = tid + i * C::NCT;
        const int rr = v < kVecs ? 4 * v / D : 0, cc = 4 * v % D;
        rp[i] = st + rr * C::REC + kRecO + cc;
        wp[i] = s_w + rr;
        O[i] = scale4(s_a[rr], O[i]);
      }
#pragma unroll 2
      for (int u = 0; u < n; ++u) {
#pragma unroll
        for (int i = 0; i < C::V4; ++i)
          O[i] = fma4(wp[i][u * kRows], *reinterpret_cast<const float4*>(rp[i] + u * C::RS), O[i]);
      }
    }
    consumer_sync(C::NCT);  // buffer bi & 1, the scalars and s_l are settled
  }
  if (!staged) *fail = true;
#pragma unroll
  for (int i = 0; i < C::V4; ++i) {
    const int v = tid + i * C::NCT;
    if (v < kVecs) Lsum[i] = s_l[4 * v / D];
  }
}

// Shared memory the shared merge of a unit of np pieces (np >= 4) needs at
// most, for any CTA's share: per-thread partial sums, per piece its share of
// O with the row headers it crosses and one weight per share row, and the
// row sums. A unit whose merge would not fit in the idle ring and merge area
// is merged at its host.
template <class C>
__host__ __device__ constexpr size_t shared_merge_bytes(int np) {
  constexpr int NV = C::MROWS * C::DIM / 4;  // vectors of 4 outputs of a unit
  const int sv = (NV + np - 2) / (np - 1);    // vectors of the largest share (at least np - 1 CTAs share)
  const int nrs = cmin(C::MROWS, (4 * sv + C::DIM - 1) / C::DIM + 1);  // record rows a share touches
  const int span = 4 * sv + 4 * (nrs - 1);    // floats of one piece's part, headers included
  return sizeof(float) * ((size_t)4 * C::NCT + (size_t)np * (span + nrs) + nrs);
}
// Whether the split unit of CTAs host .. fin is merged shared: records of
// at least kSharedMergeRows rows, at least KParams::shared_pieces pieces,
// at least kSharedMergeBytes of peer records, and room for the merge.
template <class C>
__device__ __forceinline__ bool merged_shared(const KParams& p, int host, int fin) {
  const int np = fin - host + 1;
  return C::MROWS >= kSharedMergeRows && p.shared_pieces > 0 && np >= p.shared_pieces &&
         (size_t)(np - 1) * C::RS * sizeof(float) >= kSharedMergeBytes &&
         shared_merge_bytes<C>(np) <= C::KV_BYTES + C::MERGE_BYTES;
}

// The merge of a split unit (CTAs h0 .. h1, records in slots given by
// slot()) shared by the CTAs whose last segment is one of its pieces: the
// host, the CTAs between, and the finisher when the piece is its only
// segment. Each takes an equal share of the unit's rows x d outputs (a range
// of 4-output vectors in record order), waits for every piece's ready flag,
// copies its share of each record into the idle ring (16-byte async copies,
// in flight while the row maxima and sums are read), and sums the pieces
// with the weights 2^(m_i - m) of f: the same result as folding f over the
// pieces in any order. Out of line, called after the segment loop.
template <class C>
__device__ __noinline__ void merge_unit_shared(const KParams& p, int g, int h0, int h1, int b, int kvh0, float* sm,
                                               volatile int* abort_flag, uint32_t ready) {
  constexpr int D = C::DIM, NT = C::NCT, REC = C::REC, GRP = C::MROWS / C::HPU;
  constexpr int NV = C::MROWS * D / 4;
  const int tid = threadIdx.x;
  const bool fin_last = p.cta_seg[h1 + 1] - p.cta_seg[h1] == 1;  // the finisher's piece is its only segment
  const int np = h1 - h0 + 1;
  const int npart = fin_last ? np : np - 1;
  auto slot = [&](int c) { return (c < h1 || fin_last) ? p.G + c : c; };
  // thread i waits for the flags of pieces i, i + NT, ... (not its own)
  const uint64_t twait = global_ns();
  for (int i = tid; i < np; i += NT) {
    const int c = h0 + i;
    if (c == g) continue;
    const uint32_t* f = p.flags + slot(c);
    const uint64_t tstart = global_ns();
    for (uint32_t it = 0; !*abort_flag; ++it) {
      if (ld_acquire_gpu(f) == ready) break;
      if ((it & 15u) == 15u) {
        if ((long long)(global_ns() - tstart) > p.spin_ns) {
          record_error(p.hdr, kStatusTimeout, g, c);
          *abort_flag = 1;
          break;
        }
        __nanosleep(100);
      }
    }
  }
  consumer_sync(NT);  // every flag seen (or the abort raised) before any record is read
  if (p.trace != nullptr && tid == 0) p.trace[(size_t)g * kTraceWords + kTrWaitNs] += global_ns() - twait;
  const bool fail = *abort_flag != 0;
  // this CTA's share: vectors [v0, v1), record rows rr0 .. rr0 + nrs - 1;
  // vector v sits at float off(v) of a record
  const int k = g - h0;
  const int v0 = (int)((long long)NV * k / npart), v1 = (int)((long long)NV * (k + 1) / npart);
  const int nev = v1 - v0;
  auto off = [](int v) { return (4 * v / D) * REC + kRecO + 4 * v % D; };
  const int rr0 = 4 * v0 / D;
  const int nrs = nev > 0 ? 4 * (v1 - 1) / D - rr0 + 1 : 0;
  const int a0 = off(v0), span = nev > 0 ? off(v1 - 1) + 4 - a0 : 0;
  // shared memory (the idle ring and merge area)
  float4* part4 = reinterpret_cast<float4*>(sm);  // [NT] partial weighted sums (threads splitting a vector's pieces)
  float* so = sm + 4 * NT;                        // [np][span]: every piece's part
  float* wm = so + (size_t)np * span;             // [np][nrs]: m of every piece, then its weight
  float* lr = wm + (size_t)np * nrs;              // [nrs]: the row sums l
  if (nev > 0) {
    const int q4 = span / 4;
    const uint32_t s0 = smem_u32(so);
    for (int i = tid; i < np * q4; i += NT) {
      const int pi = i / q4, c4 = i - pi * q4;
      const float* src = p.recs + (size_t)slot(h0 + pi) * C::RS + a0 + 4 * c4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s0 + 16u * (uint32_t)i), "l"(src) : "memory");
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  // one warp per share row, lane j taking pieces j, j + 32, ...: the
  // running maximum and sum of l (each m kept for the weights), combined
  // over the warp, then the weights 2^(m_i - m) of the lane's pieces; a
  // poisoned piece (NaN m) makes the row's l NaN. Rows past the unit's live
  // query rows are neither read nor stored.
  {
    const int lane = tid & 31;
    for (int ri = tid >> 5; ri < nrs; ri += NT / 32) {
      const int rr = rr0 + ri;
      if ((rr % GRP) >= p.rows) continue;  // warp-uniform
      float m = -INFINITY, l = 0.f;
      bool bad = false;
      constexpr int KB = 8;  // pieces whose loads are in flight together
      for (int p0 = lane; p0 < np; p0 += 32 * KB) {
        float mv[KB], lv[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int pi = p0 + 32 * u;
          const float* rp = p.recs + (size_t)slot(h0 + (pi < np ? pi : 0)) * C::RS + rr * REC;
          mv[u] = pi < np ? __ldcg(rp) : -INFINITY;
          lv[u] = pi < np ? __ldcg(rp + 1) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int pi = p0 + 32 * u;
          if (pi >= np) break;
          const float mi = mv[u];
          wm[pi * nrs + ri] = mi;
          bad |= mi != mi;
          if (mi > m) {
            l = (m == -INFINITY) ? 0.f : l * ex2(m - mi);
            m = mi;
          }
          if (mi > -INFINITY) l = fmaf(ex2(mi - m), lv[u], l);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(kFull, m, o), l2 = __shfl_xor_sync(kFull, l, o);
        const float mn = fmaxf(m, m2);
        l = (m == -INFINITY ? 0.f : l * ex2(m - mn)) + (m2 == -INFINITY ? 0.f : l2 * ex2(m2 - mn));
        m = mn;
      }
      bad = __any_sync(kFull, bad);
      for (int pi = lane; pi < np; pi += 32) {
        const float mi = wm[pi * nrs + ri];
        wm[pi * nrs + ri] = (mi == -INFINITY) ? 0.f : ex2(mi - m);  // NaN for a poisoned piece
      }
      if (lane == 0) lr[ri] = bad ? __int_as_float(0x7fc00000) : l;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  consumer_sync(NT);  // the weights, l and every thread's copies are in shared memory
  // the weighted sums of 4-output vectors; with fewer vectors than threads,
  // ng threads split the pieces of each vector
  const int ng = (nev >= NT || nev <= 0) ? 1 : cmin(np, NT / nev);
  const float nan = __int_as_float(0x7fc00000);
  auto store = [&](int v, float4 o) {
    const int r2 = 4 * v / D, c = 4 * v % D, hh = r2 / GRP, j = r2 % GRP;
    const float inv = 1.f / lr[r2 - rr0];
    store_out4(p.out, row_index(p, b, kvh0 + hh, j) * D + c, fail ? nan : o.x * inv, fail ? nan : o.y * inv,
               fail ? nan : o.z * inv, fail ? nan : o.w * inv, p.out_dtype);
  };
  if (ng == 1) {
    for (int v = v0 + tid; v < v1; v += NT) {
      const int r2 = 4 * v / D;
      if ((r2 % GRP) >= p.rows) continue;
      const int x = off(v) - a0, wi = r2 - rr0;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int pi = 0; pi < np; ++pi)
        o = fma4(wm[pi * nrs + wi], *reinterpret_cast<const float4*>(so + (size_t)pi * span + x), o);
      store(v, o);
    }
  } else {
    const int ei = tid % nev, jg = tid / nev;
    const int v = v0 + ei, r2 = 4 * v / D;
    const bool vlive = (r2 % GRP) < p.rows;
    if (jg < ng && vlive) {
      const int x = off(v) - a0, wi = r2 - rr0;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int pi = jg; pi < np; pi += ng)
        o = fma4(wm[pi * nrs + wi], *reinterpret_cast<const float4*>(so + (size_t)pi * span + x), o);
      part4[jg * nev + ei] = o;
    }
    consumer_sync(NT);
    if (tid < nev && vlive) {
      float4 o = part4[tid];
      for (int k2 = 1; k2 < ng; ++k2) {
        const float4 x = part4[k2 * nev + tid];
        o = make_float4(o.x + x.x, o.y + x.y, o.z + x.z, o.w + x.w);
      }
      store(v, o);
    }
  }
}

template <int D, int T, int GRP, typename E, int HP>
__device__ __forceinline__ void consume(const KParams& p, int g, E* kv, uint64_t* full, uint64_t* empty, uint64_t* stg,
                                        float* mrg, volatile int* abort_flag, uint32_t epoch) {
  using C = Cfg<D, T, GRP, HP>;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int s_begin = p.cta_seg[g], s_end = p.cta_seg[g + 1];
  const uint32_t ready = epoch + 1u;
  // Outputs of a unit: output idx -> record row rr = idx / D = hh * GRP + j
  // (kv head hh of the unit, query row j, live when j < rows) and dim idx % D.
  constexpr int kItems = HP * GRP * D;
  constexpr int kVecs = kItems / 4;  // vectors of 4 consecutive outputs
  const int groups = p.hkv / HP;  // units per request
  int stage = 0;
  uint32_t phase = 0;

  // Segment records are read one segment ahead, so a segment's record is in
  // registers when it starts.
  int4 w0n = make_int4(0, 0, 0, 0), w1n = w0n;
  if (s_begin < s_end) {
    w0n = *reinterpret_cast<const int4*>(p.segs + (size_t)s_begin * kDevSegWords);
    w1n = *reinterpret_cast<const int4*>(p.segs + (size_t)s_begin * kDevSegWords + 4);
  }
  for (int si = s_begin; si < s_end; ++si) {
    const int4 w0 = w0n, w1 = w1n;
    if (si + 1 < s_end) {
      w0n = *reinterpret_cast<const int4*>(p.segs + (size_t)(si + 1) * kDevSegWords);
      w1n = *reinterpret_cast<const int4*>(p.segs + (size_t)(si + 1) * kDevSegWords + 4);
    }
    const int unit = w0.x, t0 = w0.y, t1 = w0.z, kind = w0.w, peer = w1.x;
    const int b = unit / groups, kvh0 = (unit % groups) * HP;  // request, first kv head of the unit
    // Device offsets that disagree with the schedule: the tiles are still
    // taken from the ring (the producer streams them) but not used, and the
    // unit's outputs are NaN.
    const bool ok = unit_offsets_ok(p, b);
    if (!ok && tid == 0) record_error(p.hdr, kStatusInvalid, g, unit);
    const long long L = w1.y;
    const int n_tiles = t1 - t0;

    // ---- the LeanTile loop; leaves this warp's (m, l, O) in the merge area
    float* wrec = mrg + (size_t)warp * GRP * C::REC;
    if constexpr (C::TC)
      warp_segment_tc<D, T, GRP, E, HP>(p, g, b, kvh0, L, t0, n_tiles, ok, kv, full, empty, stage, phase,
                                        abort_flag, wrec);
    else
      warp_segment_cc<D, T, GRP, E, HP>(p, g, b, kvh0, L, t0, n_tiles, ok, kv, full, empty, stage, phase,
                                        abort_flag, wrec);
    if (p.trace != nullptr && tid == 0) {
      unsigned long long* tr = p.trace + (size_t)g * kTraceWords;
      tr[kTrTilesDone] = global_ns();
      tr[kTrSegs] += 1ull;
    }
    // Pull the next segment's query rows into L1 while this segment's
    // partial is merged and written, so the next tile loop starts without
    // a round trip to L2 for q (one 128-byte line per thread).
    if (si + 1 < s_end) {
      constexpr int kLines = (D * 2 + 127) / 128;  // lines of one query row
      if (tid < HP * p.rows * kLines) {
        const int nb = w0n.x / groups, nkvh0 = (w0n.x % groups) * HP;
        const int rr = tid / kLines, hh = rr / p.rows, j = rr % p.rows;
        const char* line = reinterpret_cast<const char*>(p.q) + row_index(p, nb, nkvh0 + hh, j) * D * 2 +
                           (tid % kLines) * 128;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(line));
      }
    }
    consumer_sync(C::NCT);

    // ---- merge the warps of each kv head with f. Each thread takes
    // vectors of 4 consecutive outputs: vector v covers record row
    // rr = 4v / D (kv head hh = rr / GRP of the unit, query row j = rr % GRP,
    // live when j < rows) and dims 4v % D .. + 3, so that records move as
    // 16-byte loads and stores (O starts 16-byte aligned in every row).
    float M[C::V4], Lsum[C::V4];
    float4 O[C::V4];
#pragma unroll
    for (int i = 0; i < C::V4; ++i) {
      const int v = tid + i * C::NCT;
      const int rr = 4 * v / D, cc = 4 * v % D, hh = rr / GRP, j = rr % GRP;
      M[i] = -INFINITY;
      Lsum[i] = 0.f;
      O[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (v < kVecs && j < p.rows) {
        const float* base = mrg + ((size_t)hh * C::WPH * GRP + j) * C::REC;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::WPH; ++w) mm = fmaxf(mm, base[w * GRP * C::REC]);
        if (mm != -INFINITY) {
          float ls = 0.f;
          float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < C::WPH; ++w) {
            const float* r = base + w * GRP * C::REC;
            const float wt = (r[0] == -INFINITY) ? 0.f : ex2(r[0] - mm);
            ls = fmaf(wt, r[1], ls);
            os = fma4(wt, *reinterpret_cast<const float4*>(r + kRecO + cc), os);
          }
          M[i] = mm;
          Lsum[i] = ls;
          O[i] = os;
        }
      }
    }
    const bool poisoned = (*abort_flag != 0) || !ok;
    // a piece of a unit whose merge every CTA ending on one of its pieces
    // shares (merge_unit_shared, after the loop): every piece writes a
    // record, the CTA's last segment in slot G + g
    const bool split = kind == kHost || kind == kNonHost;
    const bool shared =
        split && merged_shared<C>(p, kind == kHost ? g : p.segs[(size_t)si * kDevSegWords + 11], peer);

    if (kind == kNonHost || kind == kPartial || shared) {
      const int slot = (shared && si == s_end - 1) ? p.G + g : g;
      float* rec = p.recs + (size_t)slot * C::RS;
#pragma unroll
      for (int i = 0; i < C::V4; ++i) {
        const int v = tid + i * C::NCT;
        const int rr = 4 * v / D, cc = 4 * v % D;
        if (v < kVecs && rr % GRP < p.rows) {
          float* r = rec + rr * C::REC;
          *reinterpret_cast<float4*>(r + kRecO + cc) = O[i];
          if (cc == 0)
            *reinterpret_cast<float4*>(r) = make_float4(poisoned ? __int_as_float(0x7fc00000) : M[i], Lsum[i], 0.f, 0.f);
        }
      }
      // the barrier orders every thread's record stores before thread 0's
      // release store, which is cumulative at gpu scope: a CTA that
      // acquires the flag sees the whole record (no fence per thread)
      consumer_sync(C::NCT);
      if (kind != kPartial && tid == 0 && !(g == p.skip_signal && si == s_begin))
        st_release_gpu(&p.flags[slot], ready);
    } else {
      bool fail = poisoned;
      if (kind == kHost) {
        // Wait for every later CTA of the unit at once: consumer thread i
        // spins (bounded) on the ready flags of peers i, i + NCT, ...
        const int npeer = peer - g;
        const uint64_t twait = global_ns();
        for (int i = tid; i < npeer; i += C::NCT) {
          const int g2 = g + 1 + i;
          const uint64_t tstart = global_ns();
          for (uint32_t it = 0; !*abort_flag; ++it) {
            if (ld_acquire_gpu(&p.flags[g2]) == ready) break;
            if ((it & 15u) == 15u) {
              if ((long long)(global_ns() - tstart) > p.spin_ns) {
                record_error(p.hdr, kStatusTimeout, g, g2);
                *abort_flag = 1;
                break;
              }
              __nanosleep(100);
            }
          }
        }
        consumer_sync(C::NCT);  // every flag seen (or the abort raised) before any record is read
        if (p.trace != nullptr && tid == 0)
          p.trace[(size_t)g * kTraceWords + kTrWaitNs] += global_ns() - twait;
        if (*abort_flag) {
          fail = true;
        } else {
          int p0 = 0;
          if (si == s_end - 1 && npeer > C::PB) {
            host_merge_staged<C, E>(p, g, npeer, kv, stg, M, Lsum, O, &fail);
            p0 = npeer;
          }
          // Few peers (or peers beyond the staged ones): the loads of PB
          // peers for all of this thread's outputs are issued before any of
          // them is used, so a batch costs one L2 round trip.
          for (; p0 < npeer; p0 += C::PB) {
            float m2[C::V4][C::PB], l2[C::V4][C::PB];
            float4 o2[C::V4][C::PB];
#pragma unroll
            for (int i = 0; i < C::V4; ++i) {
              const int v = tid + i * C::NCT;
              const int rr = 4 * v / D, cc = 4 * v % D;
#pragma unroll
              for (int u = 0; u < C::PB; ++u) {
                m2[i][u] = -INFINITY;
                l2[i][u] = 0.f;
                o2[i][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (v < kVecs && rr % GRP < p.rows && p0 + u < npeer) {
                  const float* r = p.recs + (size_t)(g + 1 + p0 + u) * C::RS + rr * C::REC;
                  m2[i][u] = __ldcg(r);
                  l2[i][u] = __ldcg(r + 1);
                  o2[i][u] = __ldcg(reinterpret_cast<const float4*>(r + kRecO + cc));
                }
              }
            }
#pragma unroll
            for (int i = 0; i < C::V4; ++i)
#pragma unroll
              for (int u = 0; u < C::PB; ++u) merge_f4(M[i], Lsum[i], O[i], m2[i][u], l2[i][u], o2[i][u]);
          }
        }
      }
      // normalise and store: O = Obar / l
#pragma unroll
      for (int i = 0; i < C::V4; ++i) {
        const int v = tid + i * C::NCT;
        const int rr = 4 * v / D, cc = 4 * v % D;
        if (v < kVecs && rr % GRP < p.rows) {
          const float nan = __int_as_float(0x7fc00000);
          const float inv = 1.f / Lsum[i];
          store_out4(p.out, row_index(p, b, kvh0 + rr / GRP, rr % GRP) * D + cc, fail ? nan : O[i].x * inv,
                     fail ? nan : O[i].y * inv, fail ? nan : O[i].z * inv, fail ? nan : O[i].w * inv, p.out_dtype);
        }
      }
    }
    consumer_sync(C::NCT);  // the merge area is rewritten by the next segment
  }
  // The CTA's last segment, when a piece of a unit merged shared: this CTA's
  // share of the unit's outputs. Called here, after the segment loop, so
  // that no state of the loop is live across the call.
  if (s_end > s_begin) {
    const int* w = p.segs + (size_t)(s_end - 1) * kDevSegWords;
    const int kind = w[3], fin = w[4], host = w[11];
    if ((kind == kHost || kind == kNonHost) && merged_shared<C>(p, host, fin))
      merge_unit_shared<C>(p, g, host, fin, w[0] / groups, (w[0] % groups) * HP, reinterpret_cast<float*>(kv),
                           abort_flag, ready);
  }
}

// Programmatic dependent launch. Every kernel of the library first lets
// the next grid on its stream be launched (griddepcontrol.launch_dependents)
// and then waits until the grid before it has completed and its memory is
// visible (griddepcontrol.wait), before it touches global memory: launched
// with the attribute below, a kernel's CTAs can be placed on SMs as soon as
// the previous kernel's CTAs leave them, which hides the launch latency
// between back-to-back calls without reading anything early. Without a
// prerequisite grid, the wait returns at once. (The tcgen05 kernel's merge
// launch for fixed splits, thousands of small blocks, is the exception: its
// blocks, launched early, made those calls about 10 % slower.)
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// -------------------------------------------------------------------- kernel
template <int D, int T, int GRP, typename E, int HP>
__global__ void __launch_bounds__(Cfg<D, T, GRP, HP>::NTHREADS, 1)
    lean_decode_kernel(const KParams p, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  using C = Cfg<D, T, GRP, HP>;
  grid_dependency_sync();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // swizzled TMA tiles need 1024-byte aligned destinations, plain ones 128
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  E* kv = reinterpret_cast<E*>(smem);
  float* mrg = reinterpret_cast<float*>(smem + C::KV_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::KV_BYTES + C::MERGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  volatile int* flags_smem = reinterpret_cast<volatile int*>(empty + C::STAGES);  // [0] abort, [1] spare
  uint64_t* stg = empty + C::STAGES + 1;  // two barriers of the host merge's staged copies

  const int tid = threadIdx.x;
  const int g = blockIdx.x;
  if (tid == 0) {
    if (p.trace != nullptr) {
      unsigned long long* tr = p.trace + (size_t)g * kTraceWords;
      uint32_t sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      tr[kTrSm] = sm;
      tr[kTrStart] = global_ns();
      for (int w = 2; w < kTraceWords; ++w) tr[w] = 0ull;
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    mbar_init(&stg[0], 1);
    mbar_init(&stg[1], 1);
    flags_smem[0] = 0;
    flags_smem[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t epoch = *reinterpret_cast<volatile uint32_t*>(&p.hdr[kEpoch]);

  if ((tid >> 5) == C::NCW) {
    produce<C, E>(p, &tmk, &tmv, g, kv, full, empty, flags_smem);
  } else {
    consume<D, T, GRP, E, HP>(p, g, kv, full, empty, stg, mrg, flags_smem, epoch);
  }
  __syncthreads();
  if (tid == 0) {
    if (p.trace != nullptr) p.trace[(size_t)g * kTraceWords + kTrEnd] = global_ns();
    // The last CTA to finish advances the epoch, so the next launch's ready
    // flags can never be confused with this one's.
    __threadfence();
    const uint32_t prev = atomicAdd(&p.hdr[kDone], 1u);
    if (prev == (uint32_t)p.G - 1u) {
      p.hdr[kDone] = 0u;
      __threadfence();
      p.hdr[kEpoch] = epoch + 1u;
    }
  }
}

// Fixed-split baseline: merge the pieces of every unit with f (one block per
// (unit, query head of the group), one thread per dimension).
template <int D, int GRP>
__global__ void __launch_bounds__(D) lean_combine_kernel(const CParams p) {
  grid_dependency_sync();
  constexpr int REC = D + kRecO;
  const int row = blockIdx.x;  // unit * GRP + j
  const int unit = row / GRP, j = row % GRP;
  const int c = threadIdx.x;
  if (j >= p.rows) return;
  const int h0 = p.unit_host[unit], h1 = p.unit_fin[unit];
  if (h0 == h1) return;  // a whole unit was written by the decode kernel
  float M = -INFINITY, Ls = 0.f, O = 0.f;
  for (int s = h0; s <= h1; ++s) {
    const float* r = p.recs + (size_t)s * record_stride(D, GRP) + j * REC;
    const float m2 = r[0], l2 = r[1], o2 = r[kRecO + c];
    const float mn = fmaxf(M, m2);
    if (mn == -INFINITY) continue;
    const float a = (M == -INFINITY) ? 0.f : ex2(M - mn);
    const float bw = (m2 == -INFINITY) ? 0.f : ex2(m2 - mn);
    Ls = a * Ls + bw * l2;
    O = a * O + bw * o2;
    M = mn;
  }
  const int b = unit / p.hkv, kvh = unit % p.hkv;
  store_out(p.out, row_index(p, b, kvh, j) * D + c, O / Ls, p.out_dtype);
}

// ------------------------------------------------------------- host launchers
// Tensor maps of K and V seen as one [rows = hkv * total tokens, D] matrix,
// boxes of W columns x T rows, swizzled over W * 2 bytes (32, 64 or 128).
cudaError_t encode_kv_maps(const void* k, const void* v, long long rows, int d, int T, int W, int elem_type,
                           CUtensorMap* mk, CUtensorMap* mv);
// Tensor maps of a token-major or paged cache seen as [rows, hkv, d]: boxes
// of bw columns x hp heads x box_rows rows; swizzled over bw * 2 bytes when
// swizzle is set (tensor-core path), plain rows otherwise.
cudaError_t encode_kv_maps_3d(const void* k, const void* v, long long rows, int hkv, int d, int bw, int hp,
                              int box_rows, bool swizzle, int elem_type, CUtensorMap* mk, CUtensorMap* mv);

template <int D, int T, int GRP, typename E, int HP = 1>
cudaError_t launch_decode_t(const KParams& p, cudaStream_t st) {
  using C = Cfg<D, T, GRP, HP>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(lean_decode_kernel<D, T, GRP, E, HP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if (p.G <= 0) return cudaSuccess;
  CUtensorMap mk, mv;
  if (p.kv_layout != kKvSlab) {
    e = encode_kv_maps_3d(p.k, p.v, p.kv_rows, p.kv_heads, D, C::TC ? C::W : D, HP, p.box_rows, C::TC,
                          (int)Elem<E>::kTmaType, &mk, &mv);
    if (e != cudaSuccess) return e;
  } else if (HP != 1) {
    return cudaErrorInvalidValue;  // units of several kv heads read token-major or paged caches only
  } else if (C::TC) {
    e = encode_kv_maps(p.k, p.v, p.kv_rows, D, C::T, C::W, (int)Elem<E>::kTmaType, &mk, &mv);
    if (e != cudaSuccess) return e;
  } else {
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
  }
  return launch_dependent(lean_decode_kernel<D, T, GRP, E, HP>, (unsigned)p.G, C::NTHREADS, C::SMEM, st, p, mk, mv);
}

template <int D, int T, int GRP, int HP = 1>
cudaError_t capacity_t(int* per_sm) {
  using C = Cfg<D, T, GRP, HP>;
  cudaError_t e = cudaFuncSetAttribute(lean_decode_kernel<D, T, GRP, __nv_bfloat16, HP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, lean_decode_kernel<D, T, GRP, __nv_bfloat16, HP>,
                                                       C::NTHREADS, C::SMEM);
}

template <int D, int GRP>
cudaError_t launch_combine_t(const CParams& p, cudaStream_t st) {
  if (p.U <= 0) return cudaSuccess;
  return launch_dependent(lean_combine_kernel<D, GRP>, (unsigned)(p.U * GRP), D, 0, st, p);
}

}  // namespace la
