// Tensor-core partial softmax of up to 16 query rows against one chunk of
// up to 64 keys (bf16 model): the split partial (m, l, 64 weighted values)
// that attn_fold_row folds, computed with mma.sync m16n8k16 (bf16 in, fp32
// accumulate) by one warp.
//
//   S = Q K^T * 1/sqrt(64)      8 key tiles x 4 dim steps
//   m = max over visible keys, p = exp(s - m), l = sum p   (fp32)
//   a = P V                     P split as bf16 hi + lo, so the weights keep
//                               ~16 mantissa bits; 8 dim tiles x 4 key steps x 2
//
// K and V sit in shared memory as [key][64] bf16 rows of 128 bytes, either
// with the 128-byte swizzle of a TMA box (16-byte chunk c of row r at chunk
// c ^ (r & 7)) or linear; the arithmetic is the same either way.
#pragma once
#include "ws_attn_common.cuh"

__device__ __forceinline__ uint32_t smem_addr_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk c of key row r.
template <bool SWZ>
__device__ __forceinline__ uint32_t kv_off(int r, int c) {
  return (uint32_t)(r * 128 + ((SWZ ? (c ^ (r & 7)) : c) << 4));
}

// Query fragments (A operand, 16 rows x 64 dims, 4 steps of 16 dims) of rows
// q_row0 .. q_row0 + nrows - 1 of a [rows, ldq] bf16 matrix, head columns at
// col0; rows >= nrows are zero.  The loads go to L2 (rows written by other SMs).
__device__ __forceinline__ void attn_q_frags(const bf16* q, int ldq, int q_row0, int nrows, int col0,
                                             uint32_t qf[4][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int row = g + ((h & 1) ? 8 : 0);
      const int col = col0 + 16 * s + 2 * c + ((h & 2) ? 8 : 0);
      uint32_t v = 0u;
      if (row < nrows)
        v = __ldcg(reinterpret_cast<const unsigned int*>(q + (size_t)(q_row0 + row) * ldq + col));
      qf[s][h] = v;
    }
  }
}

// The chunk's partial in registers (HILO: P enters P V as bf16 hi + lo,
// ~16 mantissa bits; else as one bf16 value): lane (g = lane / 4, c = lane % 4) holds
// rows g and g + 8: (m0, l0) and acc[j][0..1] (dims 8j + 2c, + 1) for row g,
// (m1, l1) and acc[j][2..3] for row g + 8.  A row with no visible key has
// m = -inf, l = 0 and zero values.  DENSE: each row's mask is either all
// ones or empty, so the per-key tests are skipped; every row's result is
// exactly what the general path gives for the same masks.
template <bool SWZ, bool HILO = true, bool DENSE = false>
__device__ __forceinline__ void attn_chunk_regs(const uint8_t* Ks, const uint8_t* Vs, const uint32_t qf[4][4],
                                                uint64_t vis_lo, uint64_t vis_hi, float& om0, float& ol0, float& om1,
                                                float& ol1, float acc[8][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const uint32_t kb = smem_addr_u32(Ks), vb = smem_addr_u32(Vs);
  // ---- S = Q K^T: key tile j (keys 8j..8j+7), two dim steps per ldmatrix.x4
  float sc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 4; s2 += 2) {
      const int mtx = lane >> 3, rr = lane & 7;
      const int key = 8 * j + rr, chunk = 2 * s2 + mtx;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + kv_off<SWZ>(key, chunk), b0, b1, b2, b3);
      mma_bf16_16816(sc[j], qf[s2], b0, b1);
      mma_bf16_16816(sc[j], qf[s2 + 1], b2, b3);
    }
  }
  // ---- masked row maxima (rows g and g + 8), exp, row sums (quad of 4 lanes)
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = 8 * j + 2 * c + e;
      sc[j][e] *= 0.125f;                      // 1/sqrt(64)
      sc[j][2 + e] *= 0.125f;
      if (DENSE || ((vis_lo >> key) & 1ull)) m0 = fmaxf(m0, sc[j][e]);
      if (DENSE || ((vis_hi >> key) & 1ull)) m1 = fmaxf(m1, sc[j][2 + e]);
    }
  }
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
  m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
  m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = 8 * j + 2 * c + e;
      const float p0 = (DENSE || ((vis_lo >> key) & 1ull)) ? expf(sc[j][e] - m0) : 0.f;
      const float p1 = (DENSE || ((vis_hi >> key) & 1ull)) ? expf(sc[j][2 + e] - m1) : 0.f;
      sc[j][e] = p0;
      sc[j][2 + e] = p1;
      l0 += p0;
      l1 += p1;
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  // ---- a = P V with P = hi + lo (bf16 each); key step s uses key tiles 2s, 2s+1
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float* src = sc[2 * s + (h >> 1)] + ((h & 1) ? 2 : 0);
      const float x0 = src[0], x1 = src[1];
      const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
      const float2 hf = __bfloat1622float2(hi);
      ph[h] = *reinterpret_cast<const uint32_t*>(&hi);
      pl[h] = pack_bf16(x0 - hf.x, x1 - hf.y);
    }
#pragma unroll
    for (int j2 = 0; j2 < 8; j2 += 2) {
      // matrices: keys 16s+0..7 / 16s+8..15 for dims 8*j2.. and 8*(j2+1)..
      const int mtx = lane >> 3, rr = lane & 7;
      const int key = 16 * s + rr + ((mtx & 1) ? 8 : 0), chunk = j2 + (mtx >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vb + kv_off<SWZ>(key, chunk), b0, b1, b2, b3);
      mma_bf16_16816(acc[j2], ph, b0, b1);
      if (HILO) mma_bf16_16816(acc[j2], pl, b0, b1);
      mma_bf16_16816(acc[j2 + 1], ph, b2, b3);
      if (HILO) mma_bf16_16816(acc[j2 + 1], pl, b2, b3);
    }
  }
  const bool has0 = vis_lo != 0ull, has1 = vis_hi != 0ull;
  om0 = has0 ? m0 : -INFINITY;
  ol0 = has0 ? l0 : 0.f;
  om1 = has1 ? m1 : -INFINITY;
  ol1 = has1 ? l1 : 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (!has0) acc[j][0] = acc[j][1] = 0.f;
    if (!has1) acc[j][2] = acc[j][3] = 0.f;
  }
}

// One chunk: keys 0 .. 63 of Ks / Vs; the lanes' rows g and g + 8 see the
// keys whose bits are set in vis_lo / vis_hi.  Writes the partial of row r to
// part(r) (m, l, a[64]) for rows r < nrows.  Rows with no visible key get
// m = -inf, l = 0, a = 0.
template <bool SWZ, class PartPtr>
__device__ __forceinline__ void attn_chunk_partial(const uint8_t* Ks, const uint8_t* Vs, const uint32_t qf[4][4],
                                                   uint64_t vis_lo, uint64_t vis_hi, int nrows, PartPtr part) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float m0, l0, m1, l1, acc[8][4];
  attn_chunk_regs<SWZ>(Ks, Vs, qf, vis_lo, vis_hi, m0, l0, m1, l1, acc);
  if (g < nrows) {
    float* p = part(g);
    if (c == 0) { p[0] = m0; p[1] = l0; }
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<float2*>(p + 2 + 8 * j + 2 * c) = make_float2(acc[j][0], acc[j][1]);
  }
  if (g + 8 < nrows) {
    float* p = part(g + 8);
    if (c == 0) { p[0] = m1; p[1] = l1; }
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<float2*>(p + 2 + 8 * j + 2 * c) = make_float2(acc[j][2], acc[j][3]);
  }
}
