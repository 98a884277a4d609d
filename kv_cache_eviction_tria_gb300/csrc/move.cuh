// Row-move helpers of the in-place compaction, shared by the compaction
// stage (k_move) and the fused pass (k_pass): the per-warp staging layout of
// one 32-row destination block and the warp-wide gathers / stores of a plane.
#pragma once

#include "tria_internal.cuh"

namespace tria {

// One staging buffer: the moving rows of one chunk, every plane packed
// in destination order.
struct MoveStage {
  int k, ks, v, vs, pos, bytes;
};

__host__ __device__ inline MoveStage move_stage_layout(int k_rb, int ks_rb, int v_rb, int vs_rb) {
  MoveStage L;
  int off = 0;
  auto take = [&](int b) {
    const int at = off;
    off = (off + b + 15) & ~15;
    return at;
  };
  L.k = take(kChunk * k_rb);
  L.ks = take(kChunk * ks_rb);
  L.v = take(kChunk * v_rb);
  L.vs = take(kChunk * vs_rb);
  L.pos = -1;   // positions travel in registers and the warp's source-row table
  L.bytes = off;
  return L;
}

// 14 stages of fp16 key + value rows (16 KB each) with ~2.1 KB of static
// tables: under the 227 KB per CTA, and 152 x 14 warps cover the 2048
// destination blocks of a 32K-row, 8-head, 25 % layer in one round
constexpr int kMoveSmemLimit = 224 * 1024;
constexpr int kMoveMaxWarps = 16;

__host__ __device__ inline int move_warps(const MoveStage& L) {
  int w = kMoveSmemLimit / L.bytes;
  return w > kMoveMaxWarps ? kMoveMaxWarps : w;
}

// Lane -> (row, unit) mapping of one plane for the warp-wide row copies: a
// row of `rb` bytes is `per` units of `unit` bytes; when per <= 32 a warp
// instruction covers `rpi` rows, else a row takes several instructions.
struct PlaneMap {
  int rb, unit, per, rpi, lr, lu;
};

__device__ __forceinline__ PlaneMap plane_map(int rb, int lane) {
  PlaneMap m;
  m.rb = rb;
  m.unit = (rb & 15) == 0 ? 16 : ((rb & 7) == 0 ? 8 : ((rb & 3) == 0 ? 4 : 2));
  m.per = rb > 0 ? rb / m.unit : 1;
  m.rpi = m.per <= 32 ? 32 / m.per : 1;
  m.lr = m.per <= 32 ? lane / m.per : 0;
  m.lu = m.per <= 32 ? lane - m.lr * m.per : lane;
  return m;
}

__device__ __forceinline__ void copy_unit_async(uint8_t* d, const uint8_t* g, int unit) {
  if (unit == 16) cp_async16(d, g);
  else if (unit == 8) cp_async8(d, g);
  else if (unit == 4) cp_async4(d, g);
  else *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(g);
}

// gather rows src[0 .. rows) of one plane into packed staging (cp.async)
__device__ __forceinline__ void warp_gather(const uint8_t* plane, int64_t row0, const PlaneMap& m,
                                            uint8_t* stage, const int* src, int rows) {
  if (m.rb == 0 || rows == 0) return;
  if (m.per <= 32) {
    if (m.lr >= m.rpi) return;
    for (int j = m.lr; j < rows; j += m.rpi)
      copy_unit_async(stage + (size_t)j * m.rb + m.lu * m.unit,
                      plane + (size_t)(row0 + src[j]) * m.rb + m.lu * m.unit, m.unit);
  } else {
    for (int j = 0; j < rows; ++j) {
      const uint8_t* g = plane + (size_t)(row0 + src[j]) * m.rb;
      for (int u = m.lu; u < m.per; u += 32)
        copy_unit_async(stage + (size_t)j * m.rb + u * m.unit, g + u * m.unit, m.unit);
    }
  }
}

// write `rows` packed staged rows of one plane to consecutive rows from dst
__device__ __forceinline__ void warp_scatter(uint8_t* plane, int64_t row0, int rb, const uint8_t* stage, int dst,
                                             int rows, int lane) {
  if (rb == 0 || rows == 0) return;
  const size_t bytes = (size_t)rows * rb;
  uint8_t* out = plane + (size_t)(row0 + dst) * rb;
  if ((rb & 15) == 0) {
    for (size_t u = lane; u < bytes / 16; u += 32)
      reinterpret_cast<uint4*>(out)[u] = reinterpret_cast<const uint4*>(stage)[u];
  } else if ((rb & 3) == 0) {
    for (size_t u = lane; u < bytes / 4; u += 32)
      reinterpret_cast<uint32_t*>(out)[u] = reinterpret_cast<const uint32_t*>(stage)[u];
  } else {
    for (size_t u = lane; u < bytes / 2; u += 32)
      reinterpret_cast<uint16_t*>(out)[u] = reinterpret_cast<const uint16_t*>(stage)[u];
  }
}

}  // namespace tria
