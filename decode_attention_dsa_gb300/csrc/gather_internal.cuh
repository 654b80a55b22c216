// Internal interface between the hot-gather and attention translation units:
// the gather workspace layout and the classification/assignment launch. Not
// part of the C ABI.
#pragma once

#include "common.cuh"

struct GatherWs {
  int32_t* fill_pos;    // [U][RK] position of the i-th inserted miss (ascending)
  int32_t* fill_slot;   // [U][RK] its slot
  int32_t* fill_entry;  // [U][RK] entry (r*K + j) of the position's first occurrence
  int32_t* fill_of;     // [U][RK] per entry: the fill it owns (rank), or -1
  int32_t* nfill;       // [U]
  uint8_t* served;      // [U][RK] 1 if the entry's row is written by a fill
  int32_t* dup;         // [U][RK][MAX_ROWS-1] later occurrences of the i-th inserted miss
};

inline GatherWs gather_ws(void* ws, int32_t U, int32_t R, int32_t K) {
  const size_t rk = (size_t)R * K;
  const size_t a = dsa_align((size_t)U * rk * 4, 256);
  char* b = static_cast<char*>(ws);
  GatherWs g;
  g.fill_pos = reinterpret_cast<int32_t*>(b);
  g.fill_slot = reinterpret_cast<int32_t*>(b + a);
  g.fill_entry = reinterpret_cast<int32_t*>(b + 2 * a);
  g.fill_of = reinterpret_cast<int32_t*>(b + 3 * a);
  g.nfill = reinterpret_cast<int32_t*>(b + 4 * a);
  g.served = reinterpret_cast<uint8_t*>(b + 4 * a + dsa_align((size_t)U * 4, 256));
  g.dup = reinterpret_cast<int32_t*>(b + 4 * a + dsa_align((size_t)U * 4, 256) + dsa_align((size_t)U * rk, 256));
  return g;
}

// Classification, pinning and ring-replacement assignment of one gather call
// (k_assign); fills in the workspace and the map update. Returns a DSA_ status.
int dsa_launch_assign(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t round,
                      const int32_t* topk_idx, uint8_t* cls, int32_t* counters, void* ws, int32_t* dev_err,
                      cudaStream_t st);
