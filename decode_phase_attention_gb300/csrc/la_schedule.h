// la_schedule.h -- the host-side schedule behind the opaque la_schedule
// handle: the planner's tables and their device copy.
#pragma once

#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

struct la_schedule {
  int batch = 0, hq = 0, hkv = 0, d = 0, grp = 0, T = 0;
  int nq = 1;      // query tokens per request (speculative decoding: 2..8)
  int R = 0;       // query rows per unit the kernel instance holds: unit_grp() * nq rounded up to 1, 2, 4, 8 or 16
  int hp = 1;      // kv heads per unit: 1, or 2, 4, 8 for token-major / paged caches with short rows
  // Query blocks per kv head: when grp * nq query rows exceed the 16 an
  // instance holds, the grp query heads of a kv head are split into qb
  // blocks of grp / qb consecutive heads, each a unit of its own that reads
  // the kv head's K/V (hp is then 1).
  int qb = 1;
  int stages = 0;  // ring stages requested with la_schedule_set_stages (0: the library's choice)
  int kind = 0;    // 0 stream-K, 1 fixed
  int splits = 0;  // fixed partitions only
  int G = 0, U = 0;
  int64_t I = 0;
  // Number of this schedule among all schedules the process has made (from
  // 1): a table copy can be recognised even when a destroyed schedule's
  // address is reused by a new one.
  uint64_t serial = 0;
  std::vector<int32_t> cu, cta_iter, unit_iter, cta_seg, segs, unit_host, unit_fin;
  std::vector<int32_t> dev_segs;  // device records (kDevSegWords per segment)
  // debug hooks
  int skip_signal = -1;
  long long spin_ns = 2000000000LL;
  unsigned long long* trace = nullptr;  // device buffer of G * 8 words, or null
  // device copy: [cu (batch+1)] [cta_seg (G+1)] [segs] [unit_host (U)] [unit_fin (U)]
  std::mutex mu;
  int device = -1;
  int32_t* dev = nullptr;
  size_t off_cu = 0, off_cta_seg = 0, off_segs = 0, off_host = 0, off_fin = 0;

  // The kernel's view: unit_heads() heads per request of unit_grp() query
  // heads each; head h covers query heads h * unit_grp() on and is query
  // block h % qb of kv head h / qb (the kernel addresses K/V only through
  // the kv head the device segment records carry).
  int unit_heads() const { return hkv * qb; }
  int unit_grp() const { return grp / qb; }
};

// Source of la_schedule::serial.
inline uint64_t la_next_schedule_serial() {
  static std::atomic<uint64_t> next{0};
  return ++next;
}
