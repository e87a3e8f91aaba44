// la_internal.h -- what the C ABI layer and the kernels share: kernel
// parameters, the workspace layout and the launch entry points.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

// Kinds of segment (match LA_SEG_* in lean_attn.h).
enum SegKind : int32_t { kWhole = 0, kNonHost = 1, kHost = 2, kPartial = 3 };

// One segment of a CTA's work: the planner's 5 words (unit, tile_begin,
// tile_end, kind, peer) as exported, and the 8-word device record that adds
// the request's context length and the slab's first K/V row (64-bit), so the
// producer can issue its first copy after two dependent loads.
constexpr int kSegWords = 5;
// unit, t0, t1, kind, peer, L, row0 low, row0 high, cu[b], b, first kv head of the unit, host;
// for host and non-host pieces peer is the unit's finisher CTA and host its host CTA (else -1, 0)
constexpr int kDevSegWords = 12;

// Where the K/V rows of a (request, kv head, token) live.
enum KvLayout : int {
  kKvSlab = 0,        // request b: [hkv, L_b, d] slab at row hkv*cu[b] (1-D bulk copies / 2-D TMA)
  kKvTokenMajor = 1,  // [total tokens, hkv, d], token t of request b at row cu[b] + t (3-D TMA)
  kKvPaged = 2        // [pages, page_size, hkv, d] with a block table per request (3-D TMA)
};

// Workspace: a 256-byte header, ready flags (padded to 256 bytes), then
// partial records, one flag per record slot. Records of the 16-row kernel
// hold rows * (d + 4) floats (per query row [m, l, 0, 0, O[d]]; rows = the
// instance's rows per kv head x kv heads per unit). With fewer than
// kSharedMergeRows rows it has one slot per CTA: a CTA writes at most one
// record (its first segment's, when that is a non-host or fixed-split
// piece), and hosts merge their peers from registers. From
// kSharedMergeRows rows a split unit of many pieces (kSharedMergeBytes),
// and on the tcgen05 kernel (its records column-major) every split unit,
// is merged by every CTA that ends on one of its pieces, so each of
// its pieces writes a record: in slot CTA when the piece is not the CTA's
// last segment, else in slot G + CTA; such instances have two slots per
// CTA.
constexpr size_t kHeaderBytes = 256;
enum HeaderWord { kEpoch = 0, kDone = 1, kStatus = 2, kInfoCta = 3, kInfoPeer = 4 };

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t flags_bytes(int n) { return align_up(sizeof(uint32_t) * (size_t)n, 256); }
// Records of the 16-row kernel hold rows of [m, l, 0, 0, O[d]] (O 16-byte
// aligned, so that partials move as 16-byte vectors); the tcgen05 kernel's
// hold columns [m], [l], [O dim c] over the unit's rows (128-row instance),
// padded to a multiple of 4 floats.
constexpr int kRecO = 4;  // offset of O in a row of a 16-row kernel record
__host__ __device__ constexpr int record_stride(int d, int rows) { return rows * (d + kRecO); }
__host__ __device__ constexpr int record_stride_wide(int d, int rows) { return (rows * (d + 2) + 3) / 4 * 4; }
constexpr int kWideInstanceRows = 128;  // rows of the tcgen05 kernel's instance (kWideRows)
// 16-row kernel: from kSharedMergeRows record rows, a split unit of at
// least kSharedMergePieces pieces whose host would read at least
// kSharedMergeBytes of its peers' records is merged by every CTA that ends
// on one of its pieces (KParams::shared_pieces), not by its host alone.
// Below that the host's merge is as fast (same-box measurements: the shared
// merge's chain of flag, copy and sum after the last piece costs what the
// host spends on about 100 KB of records).
constexpr int kSharedMergeRows = 4;
constexpr int kSharedMergePieces = 4;
constexpr size_t kSharedMergeBytes = 96 * 1024;
inline int shared_merge_pieces(int rows) {
  return rows >= kSharedMergeRows && rows < kWideInstanceRows ? kSharedMergePieces : 0;
}
inline size_t record_floats(int d, int rows) {
  return (size_t)(rows >= kWideInstanceRows ? record_stride_wide(d, rows) : record_stride(d, rows));
}
// shared = false: the layout of a launch whose 16-row kernel merges every
// split unit at its host (KParams::shared_pieces = 0), one slot per CTA.
inline int record_slots(int G, int rows, bool shared = true) {
  return rows >= kWideInstanceRows || (shared && rows >= kSharedMergeRows) ? 2 * G : G;
}
inline size_t records_bytes(int G, int d, int rows, bool shared = true) {
  return sizeof(float) * record_floats(d, rows) * (size_t)record_slots(G, rows, shared);
}
inline size_t workspace_bytes(int G, int d, int rows, bool shared = true) {
  return kHeaderBytes + flags_bytes(record_slots(G, rows, shared)) + records_bytes(G, d, rows, shared);
}
// Byte offsets of the flags and the records inside a workspace.
struct WsLayout {
  size_t flags, recs, end;
};
inline WsLayout workspace_layout(int G, int d, int rows, bool shared = true) {
  WsLayout w;
  w.flags = kHeaderBytes;
  w.recs = w.flags + flags_bytes(record_slots(G, rows, shared));
  w.end = w.recs + records_bytes(G, d, rows, shared);
  return w;
}

struct KParams {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cu;        // device cu_seqlens_k from the caller
  const int32_t* sched_cu;  // the schedule's own copy (batch + 1)
  const int32_t* cta_seg;   // [G + 1]
  const int32_t* segs;      // [nseg * kSegWords]
  void* out;                // fp32, fp16 or bf16 per out_dtype
  uint32_t* hdr;
  uint32_t* flags;
  float* recs;
  long long kv_rows;        // hkv * total tokens: rows of K (and V) seen as [rows, d]
  int G;
  int batch;
  int hq;
  int hkv;                  // unit heads per request: kv heads x query blocks per kv head
  int kv_heads = 0;         // kv heads of the K/V tensors (token-major / paged tensor maps)
  float qscale;             // scale * log2(e): scores are kept in base-2 units
  long long spin_ns;        // limit of every wait inside the kernel
  int skip_signal;          // test hook: this CTA never sets its first segment's flag (-1: none)
  unsigned long long* trace;  // optional per-CTA timeline (kTraceWords each), or null
  int out_dtype = 0;          // 0 fp32, 1 fp16, 2 bf16
  // Query rows of a unit: rows = grp * nq (<= the instance's row count);
  // row r is query token r / grp of the request and head kvh * grp + r % grp,
  // kvh the unit head (a kv head, or one query block of one).
  int grp = 1;                // query heads per unit head
  int nq = 1;                 // query tokens per request (speculative decoding: > 1)
  int rows = 1;               // grp * nq
  int kv_layout = kKvSlab;
  const int32_t* block_table = nullptr;  // paged: [batch, bt_stride] page ids
  int bt_stride = 0;
  int page_size = 0;                     // paged: tokens per page
  int box_rows = 0;                      // 3-D TMA: token rows per load (T, or the page size if smaller)
  int stages = 0;                        // ring stages to cycle through (0: all the instance holds)
  // 16-row kernel: split units of at least this many pieces are merged by
  // every CTA that ends on one of their pieces (0: each by its host alone);
  // nonzero only with two record slots per CTA (record_slots)
  int shared_pieces = 0;
};

// Per-CTA trace record (globaltimer ns): written when KParams::trace is set.
constexpr int kTraceWords = 8;
enum TraceWord {
  kTrSm = 0,         // SM the CTA ran on
  kTrStart = 1,      // kernel entry
  kTrFirstTile = 2,  // first tile landed in shared memory
  kTrTilesDone = 3,  // last tile of the last segment consumed
  kTrWaitNs = 4,     // total time the host CTA spent waiting for ready flags
  kTrEnd = 5,        // all outputs / partials written
  kTrTiles = 6,      // LeanTiles processed
  kTrSegs = 7        // segments processed
};

struct CParams {            // fixed-split merge launch
  const int32_t* unit_host; // [U]
  const int32_t* unit_fin;  // [U]
  const float* recs;
  void* out;
  int U;
  int hq;
  int hkv;                  // unit heads per request (KParams::hkv)
  int out_dtype = 0;        // 0 fp32, 1 fp16, 2 bf16
  int grp = 1;              // query heads per unit head
  int nq = 1;               // query tokens per request
  int rows = 1;             // grp * nq
};

// LeanTile sizes: the default per head dim, and whether (d, T) is built for
// units of hp kv heads (T tokens of each head per tile).
int default_tile(int d);
// Default LeanTile of a stream-K slab-layout schedule with `rows` query rows
// per kv head: the table's size, except 64 tokens at d = 128 on the CUDA-core
// path (rows <= 2), which measured 1.1-1.3 % faster on GB300 with every SM
// busy.
int slab_tile(int d, int rows);
// Ring stages a stream-K launch over every SM uses (0: all the instance
// holds). With every SM streaming, fewer bytes in flight per SM measured
// faster at d = 96 and at d = 128 with 128-token tiles (slab and paged
// layouts); partitions with few busy SMs keep the whole ring.
int stream_stages(int d, int T, int hp, int kv_layout);
bool tile_supported(int d, int T, int hp = 1);

// Units of more than 16 query rows run on the tcgen05 kernel (la_wide.cuh),
// whose instance holds kWideRows rows, with one kv head per unit; head dims
// 64, 80, 96 and 128 with 128-token tiles and up to 128 rows, 256 with
// 64-token tiles and up to 64 rows (wide_supported, wide_tile,
// wide_max_rows).
constexpr int kWideRows = 128;
constexpr int kWideTile = 128;
bool wide_supported(int d);
int wide_tile(int d);
int wide_max_rows(int d);
cudaError_t launch_wide(int d, int dtype, const KParams& p, cudaStream_t st);
cudaError_t wide_capacity(int d, int* per_sm);
cudaError_t launch_combine_wide(int d, const CParams& p, cudaStream_t st);

// Launches (la_kernels_d<d>.cu, one file per head dim; la_kernels_d<d>_hp<h>.cu
// for units of h kv heads; grp == kWideRows: la_kernels_wide.cu). dtype: 0 fp16, 1 bf16.
// cudaErrorInvalidValue for a (d, T, grp, hp) that is not built.
cudaError_t launch_decode(int d, int T, int grp, int hp, int dtype, const KParams& p, cudaStream_t st);
cudaError_t launch_combine(int d, int grp, const CParams& p, cudaStream_t st);
// CTAs of the decode kernel one SM holds at once (cudaOccupancy...).
cudaError_t decode_capacity(int d, int T, int grp, int hp, int* per_sm);
// The same, cached per (device, d, T, grp, hp) on the host, and the current
// device's SM count (la_api.cu). Both return an la_status value (0 = LA_OK).
int cached_capacity(int d, int T, int grp, int hp, int* per_sm);
int device_sm_count(int* sms);
#define LA_DECLARE_HEAD_DIM(D)                                                           \
  cudaError_t launch_decode_d##D(int T, int grp, int dtype, const KParams& p, cudaStream_t st); \
  cudaError_t launch_combine_d##D(int grp, const CParams& p, cudaStream_t st);           \
  cudaError_t decode_capacity_d##D(int T, int grp, int* per_sm);
LA_DECLARE_HEAD_DIM(64)
LA_DECLARE_HEAD_DIM(80)
LA_DECLARE_HEAD_DIM(96)
LA_DECLARE_HEAD_DIM(128)
LA_DECLARE_HEAD_DIM(256)
#undef LA_DECLARE_HEAD_DIM
#define LA_DECLARE_HEAD_DIM_HP(D, H)                                                            \
  cudaError_t launch_decode_d##D##_hp##H(int T, int grp, int dtype, const KParams& p, cudaStream_t st); \
  cudaError_t decode_capacity_d##D##_hp##H(int T, int grp, int* per_sm);
LA_DECLARE_HEAD_DIM_HP(64, 2)
LA_DECLARE_HEAD_DIM_HP(80, 2)
LA_DECLARE_HEAD_DIM_HP(80, 8)
LA_DECLARE_HEAD_DIM_HP(96, 2)
LA_DECLARE_HEAD_DIM_HP(96, 4)
#undef LA_DECLARE_HEAD_DIM_HP

}  // namespace la
