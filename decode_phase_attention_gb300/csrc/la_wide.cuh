// la_wide.cuh -- the stream-K decode kernel for units of up to 128 query
// rows (64 at d = 256; multi-query attention, wide query-head groups, a
// group times many query tokens) on the 5th-generation tensor cores.
//
// With a whole query-head group in one unit, a LeanTile ("3.3 LeanTile" of
// the xllm-io review: S_f = Q K^T, the running max m and sum l, O_acc =
// P V + diag(rescale) O_acc) is a real matrix product: 128 query rows
// against T = 128 tokens, up to 128 flop per K/V byte. The 16-row kernel's
// mma.sync path cannot keep up with HBM there, so this kernel puts both
// products on tcgen05 with the accumulators in tensor memory (TMEM):
//
//   S = Q K^T    M = 128 query rows (spare rows are zero queries), N = T
//                tokens, K = d. A = Q in TMEM (written once per segment),
//                B = the K tile as the TMA ring holds it (K-major, 128-byte
//                swizzle).
//   O += P V     M = 128 rows, N = d, K = T. A = P in TMEM, B = the V tile
//                (d-major, i.e. MN-major, 128-byte swizzle).
//
// Warps: 0-15 the softmax warps (a TMEM lane quadrant -- 32 query rows --
// is reachable only from one SM sub-partition, so four warps share each
// quadrant, one quarter of the tile's tokens and of the head dims each);
// 16 the TMA producer (the 16-row kernel's producer warp, unchanged); 17
// the MMA warp (TMEM allocation, one thread issues every tcgen05.mma).
//
// TMEM (512 columns): NSB S buffers of T columns (3 of 128 at d = 64 and
// 80, 2 of 128 at d = 96 and 128, 2 of 64 at d = 256, whose LeanTile is 64
// tokens so that S, O and Q fit), then O (d columns), then Q (d / 2
// columns: two 16-bit values per column). At d = 256 units hold at most 64
// rows (lane replicas): a thread then holds 32 O values, the 32 dims of
// its quarter its replica owns; the rest come from tensor memory through
// shared memory in pieces of 16. The softmax of tile j reads S_j (buffer
// j % NSB), then writes P_j over it as a bf16/fp16 high part (columns
// +0 .. T/2 - 1) and low part (+T/2 .. T - 1), so that P V keeps
// fp32-level accuracy (as in the 16-row kernel). S of the next tile is computed into another buffer while the
// softmax runs; it waits only for the P V that last used that buffer.
// Keeping Q in TMEM leaves shared memory to the K/V ring (3 stages of
// 64 KiB at d = 128, 4 of 48 KiB at d = 96, 5 of 40 KiB at d = 80, 6 of
// 32 KiB at d = 64). At d = 64 and 128 the K/V boxes are 64 head dims wide
// (128-byte swizzle), at d = 96 32 dims (64-byte swizzle), at d = 80 16 dims
// (32-byte swizzle: one MMA k-step per box row; O quarters of 20 columns are
// read in pieces of 4, Q quarters of 10 written in pieces of 2). O accumulates over a
// segment's tiles in TMEM; a row's reference maximum moves only when a
// tile's maximum exceeds it by more than 2^8 (p values stay below 256), and
// only then is that row of O rescaled.
//
// Units of at most 64 rows (a second instance, NREP = 2) hold every query
// row in two lane replicas, r and r + 64, that take half of each tile's
// tokens each (P = 0 in the other half), so that all four sub-partitions
// compute 2^x; their two partial O rows are summed at the end.
//
// Partial records hold (m, l, O) per row column-major over the unit's rows
// (coalesced for a warp's 32 rows). Every piece of a split unit writes one,
// host included, and the CTAs that end on a piece of the unit each merge an
// equal share of its outputs (wide_merge_unit), so a unit split over many
// SMs is reduced by all of them rather than through its host's SM. The
// schedule, segments, ready flags with epochs, bounded waits and the abort
// protocol are the 16-row kernel's.
#pragma once

#include "la_kernel.cuh"

namespace la {

// ---------------------------------------------------------- tcgen05 wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// The warp's 32 lanes x 16 consecutive 32-bit columns: thread i gets lane
// (lane field of taddr) + i. Results are valid after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(r[0]), "r"(r[1]) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// A TMEM access of N (16, 8 or 4) consecutive columns, aligned to N.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 16) tmem_ld16(taddr, r); else if constexpr (N == 8) tmem_ld8(taddr, r); else tmem_ld4(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t* r) {
  if constexpr (N == 16) tmem_st16(taddr, r); else if constexpr (N == 8) tmem_st8(taddr, r); else tmem_st4(taddr, r);
}
// Registers written by tcgen05.ld are read only after the wait: tie them to
// it so that the compiler cannot move a use above the wait.
template <int N>
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t* r) {
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}
// Generic-proxy writes to shared memory become visible to the tensor
// cores and TMA (the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The 16 softmax warps (named barrier 1).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// Shared-memory matrix descriptor of a tcgen05 operand in a swizzled
// layout (rows of 128 or 64 bytes, 8-row atoms of 1024 or 512 bytes, atoms
// aligned to their size): start address, leading and stride byte offsets,
// the fixed version field and the swizzle mode (2: 128-byte, 4: 64-byte).
__device__ __forceinline__ uint64_t sdesc_swz(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t mode) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (mode << 61);
}
// Instruction descriptor of a dense kind::f16 MMA with fp32 accumulation:
// operand format (0 fp16, 1 bf16) for A and B, B MN-major or K-major, N, M.
template <typename E>
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return (1u << 4) | ((Elem<E>::kBf16 ? 1u : 0u) << 7) | ((Elem<E>::kBf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------ configuration
template <int D>
struct WCfg {
  static constexpr int DIM = D;
  static constexpr int HPU = 1;
  static constexpr int M = 128;                 // query rows of a unit (MMA M; TMEM lanes)
  // Rows a unit may hold: 128, or 64 at d = 256 (lane replicas only: 64 O
  // values a thread for one replica would not fit the 96 registers a
  // thread has; wider units are split into query blocks)
  static constexpr int MAX_ROWS = D == 256 ? 64 : 128;
  // LeanTile tokens (MMA N of S, K of P V): 128, or 64 at d = 256 so that
  // two S buffers, O and Q fit the 512 tensor-memory columns
  static constexpr int T = D == 256 ? 64 : 128;
  static constexpr int ROWS = T;
  static constexpr bool TC = true;              // the producer's swizzled TMA boxes
  static constexpr int W = D % 64 == 0 ? 64 : (D % 32 == 0 ? 32 : 16);  // box columns
  static constexpr int RB = W * 2;              // box row bytes: 128 (128-byte swizzle) or 64 (64-byte)
  static constexpr int NB = D / W;              // boxes per tile per tensor
  static constexpr int TILE_ELEMS = T * D;
  static constexpr int STAGE_BYTES = 2 * TILE_ELEMS * 2;
  static constexpr int BOX_BYTES = T * RB;      // one box of a K or V tile
  static constexpr int ATOM = 8 * RB;           // one 8-row swizzle atom
  static constexpr uint64_t SWZ = W == 64 ? 2 : (W == 32 ? 4 : 6);  // descriptor swizzle mode: 128, 64, 32 bytes
  static constexpr int KPB = W / 16;            // MMA k-steps (16 head dims, 32 bytes) per box row
  static constexpr int REC = D + 2;
  static constexpr int RS = record_stride_wide(D, M);
  static constexpr int NSW = 16;                // softmax warps: 4 per TMEM lane quadrant
  // partial row maxima (two tiles), partial sums of l, O quarters handed between lane replicas ([64][65])
  static constexpr int RED_BYTES = 3 * 4 * M * 4 + 64 * 65 * 4;
  static constexpr int NSB = 3 * T + D + D / 2 <= 512 ? 3 : 2;  // S / P buffers in TMEM
  static constexpr int NBARS = 2 * 6 + 3 * NSB + 2;  // full, empty (<= 6 stages), s_full, p_full, pv_done, q_ready, drain
  static constexpr int STAGES = cmin(6, (232448 - RED_BYTES - 1024 - 256) / STAGE_BYTES);
  static constexpr size_t KV_BYTES = (size_t)STAGES * STAGE_BYTES;
  // + exchange area, barriers, TMEM slot, flags; alignment slack
  static constexpr size_t SMEM = KV_BYTES + RED_BYTES + 256 + 1024;
  static constexpr int NTHREADS = NSW * 32 + 64;  // softmax warps, producer warp, MMA warp
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = NSB * T;    // S / P buffers first, then O
  static constexpr uint32_t Q_COL = O_COL + D;  // then Q
  static_assert(D == 64 || D == 80 || D == 96 || D == 128 || D == 256, "head dims of the wide kernel");
  static_assert(M == kWideInstanceRows, "record layout of the wide kernel");
  static_assert(STAGES >= 2 && SMEM <= 232448, "shared memory per CTA");
  static_assert(NBARS * 8 + 8 + 4 <= 256, "barrier area");  // barriers, TMEM slot, abort flag
  static_assert(Q_COL + D / 2 <= TMEM_COLS, "tensor memory columns");
};


// One thread's bounded wait; a wait that runs out records LA_ERR_TIMEOUT and
// raises the CTA's abort flag.
__device__ __forceinline__ bool wide_wait(const KParams& p, int g, uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag) {
  if (mbar_wait_bounded(bar, parity, abort_flag, p.spin_ns)) return true;
  if (!*abort_flag) record_error(p.hdr, kStatusTimeout, g, -1);
  *abort_flag = 1;
  return false;
}
// The same for a whole warp (the result is the same in every lane).
__device__ __forceinline__ bool wide_wait_warp(const KParams& p, int g, uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag) {
  bool ok = mbar_wait_bounded(bar, parity, abort_flag, p.spin_ns);
  ok = __all_sync(kFull, ok);
  if (!ok && (threadIdx.x & 31) == 0) {
    if (!*abort_flag) record_error(p.hdr, kStatusTimeout, g, -1);
    *abort_flag = 1;
  }
  return ok;
}

// ------------------------------------------------------------------ MMA warp
// One thread issues, for tile j of the CTA (segment by segment):
//   S_j = Q K_j^T into S buffer j % NSB, committed to s_full[j % NSB];
//   after the softmax has written P_j (p_full[j % NSB]): O (+)= P_j V_j,
//   committed to pv_done[j % NSB] and to the ring stage's empty barrier.
// S_{j+1} is issued before waiting for P_j, so the tensor cores compute the
// next scores while the softmax runs; S buffer (j+1) % NSB holds
// P_{j+1-NSB}, so that P V must be done first. Each buffer has its own
// barriers, so no wait is ever two phases behind its barrier.
template <int D, typename E>
__device__ __forceinline__ void wide_mma(const KParams& p, int g, const E* kv,
                                         uint64_t* full, uint64_t* empty, uint64_t* s_full, uint64_t* p_full,
                                         uint64_t* pv_done, uint64_t* q_ready, uint64_t* drain, uint32_t tmem,
                                         volatile int* abort_flag) {
  using C = WCfg<D>;
  constexpr uint32_t kIdS = idesc_f16<E>(C::M, C::T, false);  // A = Q, B = K tile: both K-major
  constexpr uint32_t kIdO = idesc_f16<E>(C::M, D, true);      // A = P (TMEM), B = V tile: MN-major
  const int s_begin = p.cta_seg[g], s_end = p.cta_seg[g + 1];
  const int ns = ring_stages<C>(p);
  const uint32_t kv0 = smem_u32(kv);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t j = 0;  // tiles of this CTA issued so far
  bool alive = true;

  auto issue_s = [&](uint32_t jj, int stg) {
    const uint32_t kb = kv0 + (uint32_t)stg * C::STAGE_BYTES;
    const uint32_t ds = tmem + (jj % C::NSB) * (uint32_t)C::T;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      // 16 head dims per MMA: Q columns 8 kk .. (two dims per column); the K
      // tile's box kk / KPB, 32 bytes per step into its swizzled rows
      const uint32_t ka = kb + (uint32_t)(kk / C::KPB) * C::BOX_BYTES + (uint32_t)(kk % C::KPB) * 32u;
      mma_ts(ds, tmem + C::Q_COL + 8u * (uint32_t)kk, sdesc_swz(ka, 16, C::ATOM, C::SWZ), kIdS,
             kk > 0 ? 1u : 0u);
    }
    tc_commit(&s_full[jj % C::NSB]);
  };

  for (int si = s_begin, seg = 0; si < s_end && alive; ++si, ++seg) {
    const int4 w0 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords);
    const int n_tiles = w0.z - w0.y;
    // the segment's Q rows are in shared memory and the previous segment's
    // O has been read (every MMA before this point is done)
    if (!wide_wait(p, g, q_ready, (uint32_t)seg & 1u, abort_flag)) break;
    if (!wide_wait(p, g, &full[stage], phase, abort_flag)) break;
    tc_fence_after();
    issue_s(j, stage);
    for (int t = 0; t < n_tiles; ++t) {
      const int cur = stage;
      if (++stage == ns) {
        stage = 0;
        phase ^= 1u;
      }
      if (t + 1 < n_tiles) {
        if (!wide_wait(p, g, &full[stage], phase, abort_flag) ||
            (j + 1u >= (uint32_t)C::NSB &&
             !wide_wait(p, g, &pv_done[(j + 1u - C::NSB) % C::NSB], ((j + 1u - C::NSB) / C::NSB) & 1u,
                        abort_flag))) {
          alive = false;
          break;
        }
        tc_fence_after();
        issue_s(j + 1u, stage);
      }
      if (!wide_wait(p, g, &p_full[j % C::NSB], (j / C::NSB) & 1u, abort_flag)) {
        alive = false;
        break;
      }
      tc_fence_after();
      // O (+)= P_j V_j: 16 tokens per MMA, the high and the low part of P
      const uint32_t vb = kv0 + (uint32_t)cur * C::STAGE_BYTES + (uint32_t)C::TILE_ELEMS * 2u;
      const uint32_t pc = tmem + (j % C::NSB) * (uint32_t)C::T;
#pragma unroll
      for (int kk = 0; kk < C::T / 16; ++kk) {
        // 16 tokens per step; LBO: the next W head dims (next box); SBO: the next 8 tokens
        const uint64_t vd = sdesc_swz(vb + (uint32_t)kk * 16u * C::RB, C::BOX_BYTES, C::ATOM, C::SWZ);
        mma_ts(tmem + C::O_COL, pc + 8u * (uint32_t)kk, vd, kIdO, (t > 0 || kk > 0) ? 1u : 0u);
        mma_ts(tmem + C::O_COL, pc + (uint32_t)(C::T / 2) + 8u * (uint32_t)kk, vd, kIdO, 1u);
      }
      tc_commit(&pv_done[j % C::NSB]);
      tc_commit(&empty[cur]);
      ++j;
    }
  }
  // Leave no MMA in flight: TMEM is freed after the CTA's last barrier.
  tc_commit(drain);
  volatile int no_abort = 0;
  mbar_wait_bounded(drain, 0, &no_abort, p.spin_ns);
}


// ------------------------------------------------------ merge of a split unit
// A unit split over CTAs h0 .. h1 (h0 the host: the unit's first tiles, at
// the end of its range; h1 the finisher: the unit's last tiles, at the
// start of its range) is complete only when its last piece is, at the end
// of the launch. Rather than reduce every piece through the host's SM,
// each CTA whose last segment is a piece of the unit (the host, the CTAs in
// between, and the finisher when that piece is its only segment) takes an
// equal share of the unit's rows x d outputs: it waits (bounded) for every
// other piece's ready flag, then applies f to its share: per row the
// maximum m over the pieces, the weights 2^(m_i - m) and l = sum w_i l_i,
// then per output sum w_i O_i / l. A piece's record and flag sit in its
// CTA's first slot when the piece is not that CTA's last segment, else in
// its second slot (G + CTA), so a CTA can hold both kinds at once. Every
// softmax thread passes the same named barriers; after a timeout or an
// abort the share is written as NaN.
template <int D>
__device__ __noinline__ void wide_merge_unit(const KParams& p, int g, int h0, int h1, int b, int kvh,
                                                float* sm, volatile int* abort_flag, uint32_t ready,
                                                unsigned long long* tr) {
  using C = WCfg<D>;
  constexpr int NT = C::NSW * 32;  // softmax threads
  const int tid = threadIdx.x;
  const int rows = p.rows;
  const bool fin_last = p.cta_seg[h1 + 1] - p.cta_seg[h1] == 1;  // the finisher's piece is its only segment
  const int np = h1 - h0 + 1;                                     // pieces
  const int npart = fin_last ? np : np - 1;                       // CTAs that merge a share
  auto slot = [&](int c) { return (c < h1 || fin_last) ? p.G + c : c; };
  // thread i waits for the flags of pieces i, i + 512, ...
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
  softmax_sync();  // every flag seen (or the abort raised) before any record is read
  if (tr != nullptr) tr[kTrWaitNs] += global_ns() - twait;
  const bool fail = *abort_flag != 0;
  // This CTA's share of the outputs e = c * rows + r (dim c, row r): a
  // range in the records' column-major order of O, its ends on 16-byte
  // boundaries of a record, so that each piece's part of it moves as
  // 16-byte async copies (in flight while m and l are read).
  const int E = rows * D, base = 2 * rows, k = g - h0;
  auto bound = [&](int kk) {
    if (kk <= 0) return 0;
    if (kk >= npart) return E;
    const int x = ((base + (int)((long long)E * kk / npart)) & ~3) - base;
    return x < 0 ? 0 : x;
  };
  const int e0 = bound(k), e1 = bound(k + 1), ne = e1 - e0;
  const int a0 = (base + e0) & ~3, span = ((base + e1 + 3) & ~3) - a0;  // floats of each piece's part
  // shared memory (the idle ring)
  float* so = sm;                  // [np][span]: the share's O of every piece
  float* wm = so + np * span;      // [np][rows]: m of every piece, then its weight
  float* lr = wm + np * rows;      // [rows]: the row sums l
  float* part = lr + rows;         // [2][NT]: partial results
  long long* ob = reinterpret_cast<long long*>(part + 2 * NT + ((np * (span + rows) + rows) & 1));  // [rows]: output offsets
  {
    const int q4 = span / 4;
    const uint32_t s0 = smem_u32(so);
    for (int i = tid; i < np * q4; i += NT) {
      const int pi = i / q4, c4 = i - pi * q4;
      const float* src = p.recs + (size_t)slot(h0 + pi) * C::RS + a0 + 4 * c4;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s0 + 16u * (uint32_t)i), "l"(src) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // nt threads per row r, thread j taking pieces j, j + nt, ...: the
  // running maximum and sum of l (each m kept for the weights)
  const int nt = NT / rows, r = tid % rows, jr = tid / rows;
  if (jr < nt) {
    float m = -INFINITY, l = 0.f;
    constexpr int KB = 8;  // pieces whose loads are in flight together
    for (int p0 = jr; p0 < np; p0 += KB * nt) {
      float mv[KB], lv[KB];
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        const int pi = p0 + u * nt;
        const float* rp = p.recs + (size_t)slot(h0 + (pi < np ? pi : 0)) * C::RS;
        mv[u] = pi < np ? __ldcg(rp + r) : -INFINITY;
        lv[u] = pi < np ? __ldcg(rp + rows + r) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        const int pi = p0 + u * nt;
        if (pi >= np) break;
        wm[pi * rows + r] = mv[u];
        const float mi = mv[u];
        if (mi > m) {
          l = (m == -INFINITY) ? 0.f : l * ex2(m - mi);
          m = mi;
        }
        l = fmaf((mi == -INFINITY) ? 0.f : ex2(mi - m), lv[u], l);  // NaN m (a poisoned piece) propagates
      }
    }
    part[jr * rows + r] = m;
    part[NT + jr * rows + r] = l;
  }
  softmax_sync();
  // each of the row's nt threads: the row's maximum m and l from the nt
  // partials, then the weights 2^(m_i - m) of its own pieces; the row's
  // first thread keeps l and the row's offset in the output
  if (jr < nt) {
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nt; ++j) m = fmaxf(m, part[j * rows + r]);
    for (int j = 0; j < nt; ++j) {
      const float mj = part[j * rows + r];
      l = fmaf((mj == -INFINITY) ? 0.f : ex2(mj - m), part[NT + j * rows + r], l);
    }
    for (int pi = jr; pi < np; pi += nt) {
      const float mi = wm[pi * rows + r];
      wm[pi * rows + r] = (mi == -INFINITY) ? 0.f : ex2(mi - m);
    }
    if (jr == 0) {
      lr[r] = l;
      ob[r] = (long long)row_index(p, b, kvh, r) * D;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  softmax_sync();  // the weights, l, the offsets and every thread's copies are in shared memory
  // the weighted sums; with fewer outputs than threads, ng threads split the
  // pieces of each output
  const int ng = (ne >= NT || ne <= 0) ? 1 : min(np, NT / ne);
  const float nan = __int_as_float(0x7fc00000);
  const float* sx = so + (base - a0);  // piece pi's element e at sx[pi * span + e]
  if (ng == 1) {
    for (int e = e0 + tid; e < e1; e += NT) {
      const int rr = e % rows;
      float o = 0.f;
#pragma unroll 4
      for (int pi = 0; pi < np; ++pi) o = fmaf(wm[pi * rows + rr], sx[pi * span + e], o);
      store_out(p.out, (size_t)(ob[rr] + e / rows), fail ? nan : o / lr[rr], p.out_dtype);
    }
  } else {
    const int ei = tid % ne, jg = tid / ne;
    if (jg < ng) {
      const int e = e0 + ei, rr = e % rows;
      float o = 0.f;
#pragma unroll 4
      for (int pi = jg; pi < np; pi += ng) o = fmaf(wm[pi * rows + rr], sx[pi * span + e], o);
      part[jg * ne + ei] = o;
    }
    softmax_sync();
    if (tid < ne) {
      const int e = e0 + tid, rr = e % rows;
      float o = part[tid];
      for (int k2 = 1; k2 < ng; ++k2) o += part[k2 * ne + tid];
      store_out(p.out, (size_t)(ob[rr] + e / rows), fail ? nan : o / lr[rr], p.out_dtype);
    }
  }
}

// A host whose unit has just one other piece, written by its finisher as
// that CTA's first segment (so long before this, the host's last): the host
// merges alone and from registers, without a record of its own. Thread 0
// waits (bounded) for the finisher's flag; each thread then applies f to
// its row's partial (m, l and its dims db .. db + N - 1 of O) and the
// finisher's record, and stores O / l.
template <int D, int N, int OR>
__device__ __forceinline__ void wide_sole_host(const KParams& p, int g, int fin, int b, int kvh, int row, bool live,
                                               int db, const float (&o)[OR], float m_use, float l, bool poisoned,
                                               volatile int* abort_flag, uint32_t ready, unsigned long long* tr) {
  using C = WCfg<D>;
  static_assert(N <= OR && N % 2 == 0, "dims of a thread");
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; !*abort_flag; ++it) {
      if (ld_acquire_gpu(p.flags + fin) == ready) break;
      if ((it & 15u) == 15u) {
        if ((long long)(global_ns() - t0) > p.spin_ns) {
          record_error(p.hdr, kStatusTimeout, g, fin);
          *abort_flag = 1;
          break;
        }
        __nanosleep(100);
      }
    }
    if (tr != nullptr) tr[kTrWaitNs] += global_ns() - t0;
  }
  softmax_sync();  // the flag seen (or the abort raised) before the record is read
  const bool fail = poisoned || *abort_flag != 0;
  if (!live) return;
  const int rows = p.rows;
  const float* rec = p.recs + (size_t)fin * C::RS;  // the finisher's first slot
  const float m2 = __ldcg(rec + row), l2 = __ldcg(rec + rows + row);
  const float m = fmaxf(m_use, m2);
  const float a = (m_use == -INFINITY) ? 0.f : ex2(m_use - m);
  const float w = (m2 == -INFINITY) ? 0.f : ex2(m2 - m);  // NaN m (a poisoned piece) propagates
  const float inv = 1.f / fmaf(w, l2, a * l);
  const float nan = __int_as_float(0x7fc00000);
  const size_t base = row_index(p, b, kvh, row) * D + db;
  constexpr int CH = N % 16 == 0 ? 16 : N;  // dims per batch of loads
#pragma unroll
  for (int c0 = 0; c0 < N; c0 += CH) {
    float v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) v[c] = __ldcg(rec + (size_t)(2 + db + c0 + c) * rows + row);
#pragma unroll
    for (int c = 0; c < CH; ++c) v[c] = fail ? nan : fmaf(w, v[c], a * o[c0 + c]) * inv;
    if constexpr (N % 4 == 0) {
#pragma unroll
      for (int c = 0; c < CH; c += 4) store_out4(p.out, base + c0 + c, v[c], v[c + 1], v[c + 2], v[c + 3], p.out_dtype);
    } else {
#pragma unroll
      for (int c = 0; c < CH; c += 2) store_out2(p.out, base + c0 + c, v[c], v[c + 1], p.out_dtype);
    }
  }
}

// --------------------------------------------------------- softmax warps
// Warp w (0..15) works on TMEM lane quadrant w % 4 (the lanes its SM
// sub-partition reaches): thread (w, lane) owns lane r = 32 (w % 4) + lane
// and quarter cq = w / 4 of its share of every S tile (with NREP = 1, tokens
// 32 cq .. 32 cq + 31; with NREP = 2, 16 tokens of its replica's half) and
// of O (head dims D/4 cq ..). Per segment: write the unit's Q rows to
// TMEM; per tile: read the thread's scores, mask and scale them, exchange
// the partial maxima of each row through shared memory, move the reference
// maximum if the tile's maximum exceeds it by more than 8 (base-2 units),
// write P = 2^(s - m) as high and low 16-bit parts over S, update the
// partial sum of l; at the end: add the partial sums (and, with replicas,
// the two O rows), read the O quarter and store O / l (a whole unit) or
// write the record (a piece of a split unit) and, on the CTA's last
// segment, merge this CTA's share of the unit. Every softmax thread passes the
// same named barriers, also after an abort (the waits are skipped then,
// not the barriers).
template <int D, typename E, int NREP>
__device__ __forceinline__ void wide_softmax(const KParams& p, int g, E* kv, float* red,
                                             uint64_t* full, uint64_t* s_full, uint64_t* p_full,
                                             uint64_t* pv_done, uint64_t* q_ready,
                                             uint32_t tmem, volatile int* abort_flag, uint32_t epoch) {
  using C = WCfg<D>;
  constexpr int T = C::T;
  constexpr int OQ = D / 4;  // head dims of O per thread
  constexpr int OC = OQ % 16 == 0 ? 16 : (OQ % 8 == 0 ? 8 : 4);  // O columns per TMEM access (aligned to its size)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, cq = warp >> 2;
  const int r = qd * 32 + lane;
  const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);  // this warp's 32 lanes
  // NREP = 2 (units of at most 64 rows): lanes r and r + 64 hold the same
  // query row and each replica takes half of every tile's tokens, so that
  // all four sub-partitions compute 2^x; P is zero in the other replica's
  // half, and the two O rows are summed at the end.
  constexpr int TPT = T / 4 / NREP;  // tokens of a tile per thread
  constexpr int RM = C::M / NREP;  // rows of one exchange slot
  const int half = NREP == 2 ? (qd >> 1) : 0;
  const int row = NREP == 2 ? (r & 63) : r;  // the query row lane r holds
  const int toff = NREP == 2 ? (T / 2) * half + TPT * cq : TPT * cq;        // this thread's first token
  const int tother = NREP == 2 ? (T / 2) * (1 - half) + TPT * cq : 0;      // the other replica's (P = 0)
  float* stage_o = red + 3 * 4 * C::M;  // [64][65] O quarters handed between replicas
  const int s_begin = p.cta_seg[g], s_end = p.cta_seg[g + 1];
  const uint32_t ready = epoch + 1u;
  const int ns = ring_stages<C>(p);
  float* lsum = red + 2 * 4 * C::M;  // [4][M] quarter sums of l
  int stage = 0;
  uint32_t phase = 0;
  uint32_t j = 0;  // tiles of this CTA consumed so far
  unsigned long long* tr = (p.trace != nullptr && tid == 0) ? p.trace + (size_t)g * kTraceWords : nullptr;

  for (int si = s_begin; si < s_end; ++si) {
    const int4 w0 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords);
    const int4 w1 = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords + 4);
    const int unit = w0.x, t0 = w0.y, t1 = w0.z;
    const int b = unit / p.hkv, kvh = unit % p.hkv;
    const bool ok = unit_offsets_ok(p, b);
    if (!ok && tid == 0) record_error(p.hdr, kStatusInvalid, g, unit);
    const long long L = w1.y;
    const int n_tiles = t1 - t0;
    const bool live = row < p.rows;
    const bool owner = live && half == 0;  // writes the row's record or output
    const bool warp_live = (NREP == 2 ? (qd & 1) * 32 : qd * 32) < p.rows;  // warp-uniform
    // keys the row may see in the request: its query token sits at position
    // L - nq + row / grp
    const long long lim = live ? L - (p.nq - 1 - row / p.grp) : 0;

    // ---- the unit's Q rows into TMEM (the A operand of S = Q K^T): this
    // thread's quarter of row r, two 16-bit values per column; spare rows
    // are zero
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const E*>(p.q) +
                                                        row_index(p, b, kvh, live ? row : 0) * D + (D / 4) * cq);
      uint32_t qw[D / 8];
      if constexpr (D % 32 == 0) {
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          const uint4 v = live ? src[k] : make_uint4(0u, 0u, 0u, 0u);
          qw[4 * k] = v.x;
          qw[4 * k + 1] = v.y;
          qw[4 * k + 2] = v.z;
          qw[4 * k + 3] = v.w;
        }
      } else {  // d = 80: 40 bytes of a quarter row, 8-byte aligned
        const uint2* src2 = reinterpret_cast<const uint2*>(src);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint2 v = live ? src2[k] : make_uint2(0u, 0u);
          qw[2 * k] = v.x;
          qw[2 * k + 1] = v.y;
        }
      }
      if constexpr (D / 8 == 32) {  // d = 256: 32 columns, in pieces of 16
        tmem_st16(trow + C::Q_COL + 32u * cq, qw);
        tmem_st16(trow + C::Q_COL + 32u * cq + 16u, qw + 16);
      } else if constexpr (D / 8 == 16) {
        tmem_st16(trow + C::Q_COL + 16u * cq, qw);
      } else if constexpr (D / 8 == 8) {
        tmem_st8(trow + C::Q_COL + 8u * cq, qw);
      } else if constexpr (D % 32 == 0) {  // d = 96: 12 columns, in pieces of 4 (each access aligned to its size)
#pragma unroll
        for (int k = 0; k < D / 32; ++k) tmem_st4(trow + C::Q_COL + (uint32_t)(D / 8) * cq + 4u * k, qw + 4 * k);
      } else {  // d = 80: 10 columns, in pieces of 2
#pragma unroll
        for (int k = 0; k < D / 16; ++k) tmem_st2(trow + C::Q_COL + (uint32_t)(D / 8) * cq + 2u * k, qw + 2 * k);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(q_ready);

    float m_use = -INFINITY, lq = 0.f;
    bool alive = __all_sync(kFull, *abort_flag == 0);  // warp-uniform: TMEM accesses are warp-wide
    for (int t = 0; t < n_tiles; ++t) {
      if (alive) alive = wide_wait_warp(p, g, &s_full[j % C::NSB], (j / C::NSB) & 1u, abort_flag);
      tc_fence_after();
      if (tr != nullptr) {
        if (tr[kTrFirstTile] == 0ull) tr[kTrFirstTile] = global_ns();
        tr[kTrTiles] += 1ull;
      }
      const uint32_t sc = trow + (j % C::NSB) * (uint32_t)T;
      const int tt = t0 + t;
      const bool work = alive && warp_live;
      uint32_t u[32];
      float mq = -INFINITY;
      float xs = 1.f;  // u holds scores to multiply by xs: raw (xs = qscale) or already scaled (1)
      if (work) {
        if constexpr (TPT >= 16) tmem_ld16(sc + (uint32_t)toff, u); else tmem_ld8(sc + (uint32_t)toff, u);
        if constexpr (TPT == 32) tmem_ld16(sc + (uint32_t)toff + 16u, u + 16);
        tmem_wait_ld_regs<TPT>(u);
        // visible tokens of this thread's share
        const long long lv = lim - (long long)tt * T - toff;
        const int vis = lv < 0 ? 0 : (lv > TPT ? TPT : (int)lv);
        if (vis == TPT && p.qscale > 0.f) {
          // the whole quarter is visible: the maximum of the raw scores,
          // scaled once (rounding is monotonic)
          float m0 = __uint_as_float(u[0]), m1 = __uint_as_float(u[1]);
#pragma unroll
          for (int i = 2; i < TPT; i += 2) {
            m0 = fmaxf(m0, __uint_as_float(u[i]));
            m1 = fmaxf(m1, __uint_as_float(u[i + 1]));
          }
          mq = fmaxf(m0, m1) * p.qscale;
          xs = p.qscale;
        } else {
#pragma unroll
          for (int i = 0; i < TPT; ++i) {
            const float x = i < vis ? __uint_as_float(u[i]) * p.qscale : -INFINITY;
            u[i] = __float_as_uint(x);
            mq = fmaxf(mq, x);
          }
        }
        red[(j & 1u) * 4 * C::M + (half * 4 + cq) * RM + row] = mq;
      }
      softmax_sync();  // the four quarter maxima of every row are in shared memory
      float alpha = 1.f;
      bool resc = false;
      if (work) {
        const float* rm = red + (j & 1u) * 4 * C::M + row;
        float mt = fmaxf(fmaxf(rm[0], rm[RM]), fmaxf(rm[2 * RM], rm[3 * RM]));
        if constexpr (NREP == 2) mt = fmaxf(mt, fmaxf(fmaxf(rm[4 * RM], rm[5 * RM]), fmaxf(rm[6 * RM], rm[7 * RM])));
        if (mt > m_use + 8.f) {  // move the reference maximum (always on a row's first visible tile)
          alpha = (m_use == -INFINITY) ? 0.f : ex2(m_use - mt);
          m_use = mt;
          lq *= alpha;
          resc = true;
        }
        const float nref = (m_use == -INFINITY) ? 0.f : -m_use;
        uint32_t hi[16], lo[16];
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int k = 0; k < TPT / 2; ++k) {
          // p = 2^(s - m); masked scores are -inf and give 0
          const float p0 = ex2(fmaf(__uint_as_float(u[2 * k]), xs, nref));
          const float p1 = ex2(fmaf(__uint_as_float(u[2 * k + 1]), xs, nref));
          ls0 += p0;
          ls1 += p1;
          if constexpr (Elem<E>::kBf16) {
            // high part: p truncated to bf16 (its upper 16 bits); low part:
            // the exact remainder, rounded to bf16
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            hi[k] = __byte_perm(b0, b1, 0x7632);
            lo[k] = Elem<E>::pack(p0 - __uint_as_float(b0 & 0xffff0000u), p1 - __uint_as_float(b1 & 0xffff0000u));
          } else {
            hi[k] = Elem<E>::pack(p0, p1);
            const float2 h = Elem<E>::unpack(hi[k]);
            lo[k] = Elem<E>::pack(p0 - h.x, p1 - h.y);
          }
        }
        // high parts in columns 0 .. T/2 - 1 of the buffer, low parts in
        // T/2 .. T - 1 (two 16-bit values a column)
        if constexpr (NREP == 1) {
          tmem_stn<TPT / 2>(sc + (uint32_t)(toff / 2), hi);  // this thread's TPT tokens
          tmem_stn<TPT / 2>(sc + (uint32_t)(T / 2 + toff / 2), lo);
        } else {
          const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          tmem_stn<TPT / 2>(sc + (uint32_t)(toff / 2), hi);  // this replica's tokens
          tmem_stn<TPT / 2>(sc + (uint32_t)(T / 2 + toff / 2), lo);
          tmem_stn<TPT / 2>(sc + (uint32_t)(tother / 2), zero);  // the other replica's: P = 0 in this lane
          tmem_stn<TPT / 2>(sc + (uint32_t)(T / 2 + tother / 2), zero);
        }
        lq += ls0 + ls1;
      }
      // V rows past the context: zero them, so that 0 * (whatever a cache
      // holds there) adds nothing to O
      const long long rem = L - (long long)tt * T;
      if (rem < T && alive) {
        if (mbar_wait_bounded(&full[stage], phase, abort_flag, p.spin_ns)) {  // already complete
          const int ntok = (int)rem;
          unsigned char* vt = reinterpret_cast<unsigned char*>(kv) + (size_t)stage * C::STAGE_BYTES +
                              (size_t)C::TILE_ELEMS * 2;
          const int n16 = (T - ntok) * (C::RB / 16);  // 16-byte pieces past the context in one box
          for (int i = tid; i < n16 * C::NB; i += C::NSW * 32)
            *reinterpret_cast<uint4*>(vt + (i / n16) * C::BOX_BYTES + ntok * C::RB + (i % n16) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
      }
      // a row whose reference maximum moved rescales its O quarter, once the
      // previous tile's P V is in it
      if (work && __any_sync(kFull, resc && t > 0)) {
        if (wide_wait_warp(p, g, &pv_done[(j - 1u) % C::NSB], ((j - 1u) / C::NSB) & 1u, abort_flag)) {
          tc_fence_after();
          const float a = (resc && t > 0) ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < OQ / OC; ++c) {
            uint32_t o[OC];
            const uint32_t oc = trow + C::O_COL + (uint32_t)(OQ * cq + OC * c);
            tmem_ldn<OC>(oc, o);
            tmem_wait_ld_regs<OC>(o);
#pragma unroll
            for (int k = 0; k < OC; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * a);
            tmem_stn<OC>(oc, o);
          }
        } else {
          alive = false;
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[j % C::NSB]);
      if (++stage == ns) {
        stage = 0;
        phase ^= 1u;
      }
      ++j;
    }
    if (tr != nullptr) {
      tr[kTrTilesDone] = global_ns();
      tr[kTrSegs] += 1ull;
    }

    // ---- the segment's O quarter (after its last P V) and the row sum l
    const bool have_o =
        alive && wide_wait_warp(p, g, &pv_done[(j - 1u) % C::NSB], ((j - 1u) / C::NSB) & 1u, abort_flag);
    tc_fence_after();
    // d = 256 (lane replicas only): each thread reads just the 32 dims of
    // its quarter it will own (its replica half's), so no thread holds more
    // than 32 O values; the other half's come through shared memory below
    constexpr int OR = D == 256 ? OQ / 2 : OQ;  // O values a thread holds
    float o[OR];
#pragma unroll
    for (int c = 0; c < OR; ++c) o[c] = 0.f;
    if (have_o && warp_live) {
#pragma unroll
      for (int c = 0; c < OR / OC; ++c) {
        uint32_t v[OC];
        const uint32_t oc = trow + C::O_COL + (uint32_t)(OQ * cq + (D == 256 ? OR * half : 0) + OC * c);
        tmem_ldn<OC>(oc, v);
        tmem_wait_ld_regs<OC>(v);
#pragma unroll
        for (int k = 0; k < OC; ++k) o[OC * c + k] = __uint_as_float(v[k]);
      }
    }
    tc_fence_before();
    lsum[(half * 4 + cq) * RM + row] = lq;
    softmax_sync();  // every warp's waits are over; the quarter sums are in shared memory
    // the segment's kind, finisher and host CTAs and unit head, read again
    // here rather than held in registers through the tile loop
    const int4 e0w = *reinterpret_cast<const int4*>(p.segs + (size_t)si * kDevSegWords);
    const int kind = e0w.w, fin = p.segs[(size_t)si * kDevSegWords + 4], host = p.segs[(size_t)si * kDevSegWords + 11];
    const int ub = e0w.x / p.hkv, ukvh = e0w.x % p.hkv;
    if constexpr (NREP == 1) {
      // 128-row instance (96 registers a thread): one replica owns each
      // quarter
      const float l = (lsum[row] + lsum[RM + row]) + (lsum[2 * RM + row] + lsum[3 * RM + row]);
      const bool poisoned = (*abort_flag != 0) || !ok || !have_o;
      // Records are column-major over the unit's rows (wide_rec): element
      // (col, r) at [col * rows + r], col 0 = m, 1 = l, 2 + c = O dim c, so
      // that a warp's 32 rows read and write whole 128-byte lines.
      const int rows = p.rows;
      // a host whose unit's only other piece is its finisher's first segment
      const bool sole = kind == kHost && fin == g + 1 && p.cta_seg[fin + 1] - p.cta_seg[fin] > 1;
      if (sole) {
        wide_sole_host<D, OQ>(p, g, fin, ub, ukvh, row, owner, OQ * cq, o, m_use, l, poisoned, abort_flag, ready, tr);
      } else if (kind != kWhole) {
        // a piece of a split unit: its record (the second slot when this is
        // the CTA's last segment) and its ready flag; on the CTA's last
        // segment, this CTA's share of the unit's merge follows the loop
        const bool last = si == s_end - 1;
        const int slot = (kind != kPartial && last) ? p.G + g : g;
        if (owner) {
          float* rec = p.recs + (size_t)slot * C::RS;
          if (cq == 0) {
            rec[row] = poisoned ? __int_as_float(0x7fc00000) : m_use;
            rec[rows + row] = l;
          }
  #pragma unroll
          for (int c = 0; c < OQ; ++c) rec[(size_t)(2 + OQ * cq + c) * rows + row] = o[c];
        }
        // the CTA barrier orders every thread's record stores before thread
        // 0's release store, which is cumulative at gpu scope: a CTA that
        // acquires the flag sees the whole record (no fence per thread)
        softmax_sync();
        if (kind != kPartial && tid == 0 && !(g == p.skip_signal && si == p.cta_seg[g]))
          st_release_gpu(&p.flags[slot], ready);
      } else if (owner) {  // a whole unit: normalise and store O = Obar / l
        const size_t base = row_index(p, ub, ukvh, row) * D + OQ * cq;
        const float inv = 1.f / l;
        const float nan = __int_as_float(0x7fc00000);
  #pragma unroll
        for (int c = 0; c < OQ; c += 4)
          store_out4(p.out, base + c, poisoned ? nan : o[c] * inv, poisoned ? nan : o[c + 1] * inv,
                     poisoned ? nan : o[c + 2] * inv, poisoned ? nan : o[c + 3] * inv, p.out_dtype);
      }
    } else {
      float l = (lsum[row] + lsum[RM + row]) + (lsum[2 * RM + row] + lsum[3 * RM + row]);
      // The dims of the O quarter this thread owns from here on: with lane
      // replicas the two halves split the quarter (each adds the other
      // replica's partial O row for its half), so that all 16 warps share the
      // record write and the stores; without, the whole
      // quarter.
      constexpr int NO = OQ / NREP;
      const int db = OQ * cq + (NREP == 2 ? NO * half : 0);  // first dim this thread owns
      if constexpr (NREP == 2) {
        l += (lsum[4 * RM + row] + lsum[5 * RM + row]) + (lsum[6 * RM + row] + lsum[7 * RM + row]);
        if constexpr (D == 256) {
          // each half already holds its own 32 dims in o[0, 32); the other
          // half's partial for them comes from its tensor memory in pieces
          // of 16 (pass rnd: half 1 - rnd gives, half rnd receives)
  #pragma unroll
          for (int rnd = 0; rnd < 2; ++rnd)
  #pragma unroll
            for (int ch = 0; ch < NO / 16; ++ch) {
              if (half != rnd && have_o && warp_live) {
                uint32_t v[16];
                tc_fence_after();
                tmem_ld16(trow + C::O_COL + (uint32_t)(OQ * cq + NO * rnd + 16 * ch), v);
                tmem_wait_ld_regs<16>(v);
  #pragma unroll
                for (int k = 0; k < 16; ++k) stage_o[row * 65 + cq * 16 + k] = __uint_as_float(v[k]);
              }
              softmax_sync();
              if (half == rnd) {
  #pragma unroll
                for (int k = 0; k < 16; ++k) o[16 * ch + k] += stage_o[row * 65 + cq * 16 + k];
              }
              softmax_sync();
            }
        } else {
          // first pass: the replica in lanes 64..127 hands dims [0, NO) of
          // its quarter to the one in 0..63; second pass: the other way,
          // dims [NO, OQ)
  #pragma unroll
          for (int rnd = 0; rnd < 2; ++rnd) {
            if (half != rnd) {
  #pragma unroll
              for (int k = 0; k < NO; ++k) stage_o[row * 65 + cq * 16 + k] = o[NO * rnd + k];
            }
            softmax_sync();
            if (half == rnd) {
  #pragma unroll
              for (int k = 0; k < NO; ++k) o[NO * rnd + k] += stage_o[row * 65 + cq * 16 + k];
            }
            softmax_sync();
          }
  #pragma unroll
          for (int k = 0; k < NO; ++k) o[k] = half ? o[NO + k] : o[k];  // this thread's dims into o[0, NO)
        }
      }
      const bool poisoned = (*abort_flag != 0) || !ok || !have_o;
      // Records are column-major over the unit's rows (wide_rec): element
      // (col, r) at [col * rows + r], col 0 = m, 1 = l, 2 + c = O dim c, so
      // that a warp's 32 rows read and write whole 128-byte lines.
      const int rows = p.rows;
      const bool sole = kind == kHost && fin == g + 1 && p.cta_seg[fin + 1] - p.cta_seg[fin] > 1;  // as above
      if (sole) {
        wide_sole_host<D, NO>(p, g, fin, ub, ukvh, row, live, db, o, m_use, l, poisoned, abort_flag, ready, tr);
      } else if (kind != kWhole) {
        // a piece of a split unit: its record and its ready flag (as above)
        const bool last = si == s_end - 1;
        const int slot = (kind != kPartial && last) ? p.G + g : g;
        if (live) {
          float* rec = p.recs + (size_t)slot * C::RS;
          if (owner && cq == 0) {
            rec[row] = poisoned ? __int_as_float(0x7fc00000) : m_use;
            rec[rows + row] = l;
          }
  #pragma unroll
          for (int c = 0; c < NO; ++c) rec[(size_t)(2 + db + c) * rows + row] = o[c];
        }
        // the CTA barrier orders every thread's record stores before thread
        // 0's release store, which is cumulative at gpu scope: a CTA that
        // acquires the flag sees the whole record (no fence per thread)
        softmax_sync();
        if (kind != kPartial && tid == 0 && !(g == p.skip_signal && si == p.cta_seg[g]))
          st_release_gpu(&p.flags[slot], ready);
      } else if (live) {  // a whole unit: normalise and store this thread's dims
        const size_t base = row_index(p, ub, ukvh, row) * D + db;
        const float inv = 1.f / l;
        const float nan = __int_as_float(0x7fc00000);
        if constexpr (NO % 4 == 0) {
  #pragma unroll
          for (int c = 0; c < NO; c += 4)
            store_out4(p.out, base + c, poisoned ? nan : o[c] * inv, poisoned ? nan : o[c + 1] * inv,
                       poisoned ? nan : o[c + 2] * inv, poisoned ? nan : o[c + 3] * inv, p.out_dtype);
        } else {  // d = 80: 10 dims per half
  #pragma unroll
          for (int c = 0; c < NO; c += 2)
            store_out2(p.out, base + c, poisoned ? nan : o[c] * inv, poisoned ? nan : o[c + 1] * inv, p.out_dtype);
        }
      }
    }
    softmax_sync();  // the quarter sums are rewritten by the next segment
  }
  // The CTA's last segment, when a piece of a split unit that it does not
  // merge alone: this CTA's share of the unit's merge. Called here, after
  // the segment loop, so that no state of the loop is live across the call.
  if (s_end > s_begin) {
    const int sl = s_end - 1;
    const int* w = p.segs + (size_t)sl * kDevSegWords;
    const int kind = w[3], fin = w[4], host = w[11];
    const bool sole = kind == kHost && fin == g + 1 && p.cta_seg[fin + 1] - p.cta_seg[fin] > 1;
    if ((kind == kHost || kind == kNonHost) && !sole)
      wide_merge_unit<D>(p, g, host, fin, w[0] / p.hkv, w[0] % p.hkv, reinterpret_cast<float*>(kv), abort_flag, ready,
                         tr);
  }
}

// -------------------------------------------------------------------- kernel
// NREP = 2 for units of at most 64 rows (lane replicas), 1 otherwise: two
// instances, so that each gets its own register allocation.
template <int D, typename E, int NREP>
__global__ void __launch_bounds__(WCfg<D>::NTHREADS, 1)
    lean_wide_kernel(const KParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using C = WCfg<D>;
  grid_dependency_sync();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  E* kv = reinterpret_cast<E*>(smem);
  float* red = reinterpret_cast<float*>(smem + C::KV_BYTES);  // [2][4][M] quarter maxima, [4][M] quarter sums
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::KV_BYTES + C::RED_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* s_full = empty + C::STAGES;
  uint64_t* p_full = s_full + C::NSB;
  uint64_t* pv_done = p_full + C::NSB;
  uint64_t* q_ready = pv_done + C::NSB;
  uint64_t* drain = q_ready + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  // [0] the CTA's abort flag
  volatile int* flags_smem = reinterpret_cast<volatile int*>(tslot + 2);

  const int tid = threadIdx.x, warp = tid >> 5;
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
      mbar_init(&empty[s], 1);  // one tcgen05.commit per tile
    }
    for (int b2 = 0; b2 < C::NSB; ++b2) {
      mbar_init(&s_full[b2], 1);
      mbar_init(&p_full[b2], C::NSW * 32);
      mbar_init(&pv_done[b2], 1);
    }
    mbar_init(q_ready, C::NSW * 32);
    mbar_init(drain, 1);
    flags_smem[0] = 0;
    fence_mbar_init();
  }
  if (warp == C::NSW + 1) {
    tmem_alloc(tslot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
  const uint32_t epoch = *reinterpret_cast<volatile uint32_t*>(&p.hdr[kEpoch]);

  if (warp < C::NSW) {
    wide_softmax<D, E, NREP>(p, g, kv, red, full, s_full, p_full, pv_done, q_ready, tmem, flags_smem, epoch);
  } else if (warp == C::NSW) {
    produce<C, E>(p, &tmk, &tmv, g, kv, full, empty, flags_smem);
  } else if ((tid & 31) == 0) {
    wide_mma<D, E>(p, g, kv, full, empty, s_full, p_full, pv_done, q_ready, drain, tmem, flags_smem);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::NSW + 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (tid == 0) {
    if (p.trace != nullptr) p.trace[(size_t)g * kTraceWords + kTrEnd] = global_ns();
    // The last CTA to finish advances the epoch (as in the 16-row kernel).
    __threadfence();
    const uint32_t prev = atomicAdd(&p.hdr[kDone], 1u);
    if (prev == (uint32_t)p.G - 1u) {
      p.hdr[kDone] = 0u;
      __threadfence();
      p.hdr[kEpoch] = epoch + 1u;
    }
  }
}

// Fixed-split merge of the wide kernel's records (column-major over the
// unit's rows): one block per (unit, query row), one thread per dimension.
template <int D>
__global__ void __launch_bounds__(D) lean_wide_combine_kernel(const CParams p) {
  using C = WCfg<D>;
  const int unit = blockIdx.x / C::M, j = blockIdx.x % C::M;
  const int c = threadIdx.x;
  const int rows = p.rows;
  if (j >= rows) return;
  const int h0 = p.unit_host[unit], h1 = p.unit_fin[unit];
  if (h0 == h1) return;  // a whole unit was written by the decode kernel
  // f over all pieces at once: the maximum m, then the weighted sums of l
  // and O (independent loads, several pieces in flight)
  float M = -INFINITY;
#pragma unroll 8
  for (int s2 = h0; s2 <= h1; ++s2) M = fmaxf(M, __ldcg(p.recs + (size_t)s2 * C::RS + j));
  float Ls = 0.f, O = 0.f;
  if (M != -INFINITY) {
#pragma unroll 8
    for (int s2 = h0; s2 <= h1; ++s2) {
      const float* r = p.recs + (size_t)s2 * C::RS;
      const float m2 = __ldcg(r + j);
      const float wt = (m2 == -INFINITY) ? 0.f : ex2(m2 - M);  // NaN m (poisoned) propagates
      Ls = fmaf(wt, __ldcg(r + rows + j), Ls);
      O = fmaf(wt, __ldcg(r + (size_t)(2 + c) * rows + j), O);
    }
  }
  const int b = unit / p.hkv, kvh = unit % p.hkv;
  store_out(p.out, row_index(p, b, kvh, j) * D + c, O / Ls, p.out_dtype);
}

// ------------------------------------------------------------ host launchers
template <int D, typename E>
cudaError_t launch_wide_t(const KParams& p, cudaStream_t st) {
  using C = WCfg<D>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    if constexpr (C::MAX_ROWS > 64) {
      e = cudaFuncSetAttribute(lean_wide_kernel<D, E, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
      if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(lean_wide_kernel<D, E, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if (p.G <= 0) return cudaSuccess;
  CUtensorMap mk, mv;
  if (p.kv_layout != kKvSlab)
    e = encode_kv_maps_3d(p.k, p.v, p.kv_rows, p.kv_heads, D, C::W, 1, p.box_rows, true, (int)Elem<E>::kTmaType,
                          &mk, &mv);
  else
    e = encode_kv_maps(p.k, p.v, p.kv_rows, D, C::T, C::W, (int)Elem<E>::kTmaType, &mk, &mv);
  if (e != cudaSuccess) return e;
  if (p.rows > C::MAX_ROWS) return cudaErrorInvalidValue;  // the planner splits wider units into query blocks
  // The merge of a split unit of np pieces over npart >= np - 1 CTAs holds,
  // in the ring, each piece's part of a share (at most rows x d / npart +
  // 12 floats) and m of every row, plus 4 rows + 2 x 512 + 2 floats; the total is
  // convex in np, so it is largest at np = 2 or np = G.
  {
    const size_t outs = (size_t)p.rows * D;
    auto need = [&](size_t np, size_t npart) {
      return (np * ((outs + npart - 1) / npart + 12 + p.rows) + 4 * (size_t)p.rows + 2 + 2 * C::NSW * 32) * sizeof(float);
    };
    if (need(2, 1) > C::KV_BYTES || (p.G > 2 && need((size_t)p.G, (size_t)p.G - 1) > C::KV_BYTES))
      return cudaErrorInvalidValue;
  }
  if constexpr (C::MAX_ROWS > 64) {
    if (p.rows > 64) {
      return launch_dependent(lean_wide_kernel<D, E, 1>, (unsigned)p.G, C::NTHREADS, C::SMEM, st, p, mk, mv);
    }
  }
  return launch_dependent(lean_wide_kernel<D, E, 2>, (unsigned)p.G, C::NTHREADS, C::SMEM, st, p, mk, mv);
}

template <int D>
cudaError_t launch_wide_combine_t(const CParams& p, cudaStream_t st) {
  if (p.U <= 0) return cudaSuccess;
  lean_wide_combine_kernel<D><<<p.U * WCfg<D>::M, D, 0, st>>>(p);  // an ordinary launch: see launch_dependent
  return cudaGetLastError();
}

template <int D>
cudaError_t wide_capacity_t(int* per_sm) {
  using C = WCfg<D>;
  constexpr int kRep = C::MAX_ROWS > 64 ? 1 : 2;  // an instance the head dim builds
  cudaError_t e = cudaFuncSetAttribute(lean_wide_kernel<D, __nv_bfloat16, kRep>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, lean_wide_kernel<D, __nv_bfloat16, kRep>, C::NTHREADS,
                                                       C::SMEM);
}

}  // namespace la
