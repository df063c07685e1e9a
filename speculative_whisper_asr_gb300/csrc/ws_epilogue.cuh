// GEMM epilogues: what happens to an fp32 accumulator pair (row r, features
// n and n+1).  Shared by the SIMT and the tcgen05 GEMM engines so both store
// identical results for identical accumulators.
#pragma once
#include "ws_internal.cuh"

template <typename T>
__device__ __forceinline__ float bias_at(const void* b, int n) {
  return b ? to_f<T>(reinterpret_cast<const T*>(b)[n]) : 0.0f;
}

// RoPE (RoFormer, interleaved pairs): rotate (y0, y1) = features (n, n+1) of
// a head by the angle of pair (n % 64) / 2 at absolute position pos.
__device__ __forceinline__ void rope_pair(const float* tab, int pos, int n, float& y0, float& y1) {
  const float* cs = tab + ((size_t)pos * (WS_DH / 2) + (n % WS_DH) / 2) * 2;
  float c = cs[0], s = cs[1];
  float a = y0, b = y1;
  y0 = a * c - b * s;
  y1 = a * s + b * c;
}

// n is even; features n and n+1 are both < N.  `z` is the batch index
// (request) for CROSSKV, whose rows are frame indices of that request.
// `kind` is e.kind, or the same value as a compile-time constant in a kernel
// compiled for one epilogue kind (the other cases then drop out).
template <typename T>
__device__ __forceinline__ void epi_pair(int kind, const Epi& e, int r, int n, float y0, float y1, int z) {
  switch (kind) {
    case EPI_STORE:
    case EPI_GELU: {
      float v0 = y0 + bias_at<T>(e.bias, n), v1 = y1 + bias_at<T>(e.bias, n + 1);
      if (kind == EPI_GELU) { v0 = gelu_erf(v0); v1 = gelu_erf(v1); }
      T* o = reinterpret_cast<T*>(e.out) + (size_t)r * e.ldo + n;
      o[0] = from_f<T>(v0); o[1] = from_f<T>(v1);
      break;
    }
    case EPI_F32: {
      float* o = reinterpret_cast<float*>(e.out) + (size_t)r * e.ldo + n;
      o[0] = y0 + bias_at<T>(e.bias, n); o[1] = y1 + bias_at<T>(e.bias, n + 1);
      break;
    }
    case EPI_RESID: {
      float* x = e.resid + (size_t)r * e.ldr + n;
      // L2 loads: in the persistent kernel the residual was last written by another SM
      float v0 = __ldcg(x) + (y0 + bias_at<T>(e.bias, n));
      float v1 = __ldcg(x + 1) + (y1 + bias_at<T>(e.bias, n + 1));
      x[0] = v0; x[1] = v1;
      if (e.hist) {
        int slot, j, pos;
        row_info(e.rm, r, slot, j, pos);
        float* h = e.hist + (((size_t)slot * e.max_block + j) * e.n_hist + e.hist_idx) * e.d + n;
        h[0] = v0; h[1] = v1;
      }
      break;
    }
    case EPI_QKV:
    case EPI_QKV_DRAFT: {
      int part = n / e.d, nn = n - part * e.d;
      int slot, j, pos;
      bool valid = row_info(e.rm, r, slot, j, pos);
      if (part == 0) {
        y0 += bias_at<T>(e.bias, nn); y1 += bias_at<T>(e.bias, nn + 1);
        if (kind == EPI_QKV_DRAFT) rope_pair(e.rope, min(pos, e.rm.max_pos - 1), nn, y0, y1);
        T* o = reinterpret_cast<T*>(e.out) + (size_t)r * e.d + nn;
        o[0] = from_f<T>(y0); o[1] = from_f<T>(y1);
      } else {
        if (part == 2) { y0 += bias_at<T>(e.bias2, nn); y1 += bias_at<T>(e.bias2, nn + 1); }
        if (kind == EPI_QKV_DRAFT) {
          if (part == 1) rope_pair(e.rope, min(pos, e.rm.max_pos - 1), nn, y0, y1);
          T* o = reinterpret_cast<T*>(part == 1 ? e.kout : e.vout) + (size_t)r * e.d + nn;
          o[0] = from_f<T>(y0); o[1] = from_f<T>(y1);
        } else if (valid) {
          T* o = kv_ptr<T>(e.kv, slot, pos, part - 1, nn / WS_DH) + (nn % WS_DH);
          o[0] = from_f<T>(y0); o[1] = from_f<T>(y1);
        }
      }
      break;
    }
    case EPI_HISTKV: {
      int part = n / e.d, nn = n - part * e.d;
      int slot, j, pos;
      if (!row_info(e.rm, r, slot, j, pos)) break;
      if (part == 0) rope_pair(e.rope, pos, nn, y0, y1);
      else { y0 += bias_at<T>(e.bias2, nn); y1 += bias_at<T>(e.bias2, nn + 1); }
      T* o = kv_ptr<T>(e.kv, slot, pos, part, nn / WS_DH) + (nn % WS_DH);
      o[0] = from_f<T>(y0); o[1] = from_f<T>(y1);
      break;
    }
    case EPI_CROSSKV: {
      int part = n / e.d, nn = n - part * e.d;
      if (part == 1) { y0 += bias_at<T>(e.bias2, nn); y1 += bias_at<T>(e.bias2, nn + 1); }
      int slot = e.req_ids[z];
      T* o = xkv_ptr<T>(e.xkv, slot, e.xlayer, part, nn / WS_DH, r) + (nn % WS_DH);
      o[0] = from_f<T>(y0); o[1] = from_f<T>(y1);
      break;
    }
    default:
      break;
  }
}

template <typename T>
__device__ __forceinline__ void epi_pair(const Epi& e, int r, int n, float y0, float y1, int z) {
  epi_pair<T>(e.kind, e, r, n, y0, y1, z);
}

// LM head value of one logit: suppressed ids become -inf (Whisper-Flash
// Appendix A.4: draft and target logits get the same token suppression).
__device__ __forceinline__ float epi_logit(const Epi& e, int n, float y) {
  if (e.suppress && ((e.suppress[n >> 5] >> (n & 31)) & 1u)) return -INFINITY;
  return y;
}

// Epilogue of 16 accumulator columns held by one warp: lane l holds feature
// n (consecutive across the warp) and v[c] is its value for row t + c.
// LOGITS reduces each row's (value, id) key over the warp before one
// atomicMax; the other kinds pair features (n, n + 1) through a shuffle.
// Only columns c_lo <= c < c_hi are stored.
__device__ __forceinline__ void epi_columns16(int kind, const Epi& e, int N, int t, int n, int M, int z, const float* v,
                                              int c_lo = 0, int c_hi = 16) {
  const int lane = threadIdx.x & 31;
  const int mc = min(M, t + c_hi), m0 = t + c_lo;     // rows m0 <= r < mc
  if (kind == EPI_LOGITS) {
    const bool ok = n < N;
    const bool sup = ok && e.suppress && ((e.suppress[n >> 5] >> (n & 31)) & 1u);   // one lookup per feature
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int r = t + c;
      if (r < m0 || r >= mc) continue;              // the same row for every lane
      const float y = ok && !sup ? v[c] : -INFINITY;
      if (ok && e.logits) e.logits[(long long)r * e.ldl + n] = y;
      if (e.amax) {
        // The warp's largest value, then the lowest lane holding it (the
        // lanes' ids are consecutive): for finite and infinite logits this is
        // the key a reduction of (value, id) keys gives, -0 tying with +0.
        float m = y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const unsigned hit = __ballot_sync(0xffffffffu, ok && y == m);
        if (hit && lane == __ffs(hit) - 1) atomicMax(e.amax + r, argmax_key(m, n));
      }
    }
    return;
  }
  if (kind == EPI_RESID) {
    // residual update: the 8 (row, feature pair) residual values of this lane
    // are loaded together (one L2 round trip), then x += y + b as in epi_pair
    const int odd = lane & 1, nn = n - odd;
    const float b0 = bias_at<bf16>(e.bias, nn), b1 = bias_at<bf16>(e.bias, nn + 1);
    float2 xr[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const int r = t + c + odd;
      if (r >= m0 && r < mc && nn + 1 < N) xr[c / 2] = __ldcg(reinterpret_cast<const float2*>(e.resid + (size_t)r * e.ldr + nn));
    }
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const float pc0 = __shfl_xor_sync(0xffffffffu, v[c], 1);
      const float pc1 = __shfl_xor_sync(0xffffffffu, v[c + 1], 1);
      const int r = t + c + odd;
      const float y0 = odd ? pc1 : v[c], y1 = odd ? v[c + 1] : pc0;
      if (r >= m0 && r < mc && nn + 1 < N) {
        const float v0 = xr[c / 2].x + (y0 + b0), v1 = xr[c / 2].y + (y1 + b1);
        *reinterpret_cast<float2*>(e.resid + (size_t)r * e.ldr + nn) = make_float2(v0, v1);
        if (e.hist) {
          int slot, j, pos;
          row_info(e.rm, r, slot, j, pos);
          float* h = e.hist + (((size_t)slot * e.max_block + j) * e.n_hist + e.hist_idx) * e.d + nn;
          h[0] = v0; h[1] = v1;
        }
      }
    }
    return;
  }
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float pc0 = __shfl_xor_sync(0xffffffffu, v[c], 1);
    const float pc1 = __shfl_xor_sync(0xffffffffu, v[c + 1], 1);
    if ((lane & 1) == 0) {
      const int r = t + c;
      if (r >= m0 && r < mc && n + 1 < N) epi_pair<bf16>(kind, e, r, n, v[c], pc0, z);
    } else {
      const int r = t + c + 1;
      if (r >= m0 && r < mc && n < N) epi_pair<bf16>(kind, e, r, n - 1, pc1, v[c + 1], z);
    }
  }
}
