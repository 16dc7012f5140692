// hp_host.h -- host-side helpers shared by the C ABI (hp_api.cu) and the
// planner (hp_plan.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include "hp_internal.h"

namespace hp {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool supported_d(int d) { return d == 64 || d == 128; }

// A tensor-core item processes at most kMaxTcTiles 128-key tiles.
constexpr int64_t kMaxTcTiles = 128;

// SMs of the current device (152 when none can be queried).
int device_sms();

// Paged pool [num_pages][Hkv][ps][d], 128-byte swizzle: bf16, box = 64
// columns x box_tok tokens x box_heads heads; or (e4m3) one byte per element,
// box = d (128) bytes x box_tok tokens x box_heads heads.
bool encode_pool_map(CUtensorMap *m, const void *pool, int num_pages, int Hkv, int ps, int d, int box_tok,
                     int box_heads = 1, bool e4m3 = false);

// The step's workspace: status word, partial LSE [rows] f32, partial O
// [rows][d] bf16.
struct WsLayout {
    size_t off_lse, off_o, total;
};
WsLayout ws_layout(int64_t part_rows, int d);

}  // namespace hp
