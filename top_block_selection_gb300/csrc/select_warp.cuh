// select_warp.cuh - exact top-k of one score row by ONE warp, for k <= 128
// (Strata pull request 228, part 1, and pull request 856 "Arithmetic contract
// and parity": the top-k over the block scores with a block-index tie-break).
//
// Same order as select_row.cuh: descending score, equal scores by ascending
// block index, -0.0 == +0.0, ids past min(k, nb) are -1. Keys are the
// order-preserving uint32 score keys; a winner is the 64-bit value
// (key << 32 | ~index), all distinct, larger = earlier in the output.
//
// No barrier wider than the warp, so an SM can hold as many rows in flight as
// it has warps: the form for launches of many rows (a prefill's selection),
// where the group selects of select_row.cuh are bound by the latency of their
// barrier-separated phases.
//   1. threshold: the keys are cut into 128 segments (key index mod 128) and
//      each segment's maximum taken. With kk = min(k, nb) <= 128 segments
//      non-empty, the kk-th largest of those maxima, T, is a lower bound of
//      the kk-th largest key (kk distinct keys, the maxima, are >= T), so
//      every winner has key >= T. The 128 maxima are sorted by the warp
//      bitonic network (4 per lane).
//   2. candidates: the keys >= T (about 1.2-1.5 k on score rows) are
//      compacted into the warp's buffer by a count pass, a warp scan and a
//      write pass.
//   3. up to 256 candidates are sorted by the warp bitonic network on their
//      64-bit winner values (4 or 8 per lane); the first kk are the output.
//   Otherwise (mass ties or flat rows: more than 256 keys >= T) the kk-th
//   largest key value v is found by bisection between T and the maximum, the
//   keys above v are taken with the (kk - #above) smallest-index keys equal
//   to v, and those kk winners are sorted.
#pragma once

#include "qsa_device.cuh"
#include "select_row.cuh"

namespace qsa {

constexpr int kWarpSelKMax = 128;  // k the warp select handles
constexpr int kWarpSelCap = 256;   // candidates sorted in registers

// Warp bitonic network: sorts the warp's 32 E values descending in place,
// element e = lane * E + j in v[j] of lane e / E. Blocks of size s are built
// descending where (e & s) == 0 and ascending otherwise, so the last stage
// (s = 32 E) leaves the whole warp descending.
template <int E, typename V>
__device__ __forceinline__ void warp_bitonic_desc(V (&v)[E], int lane) {
  constexpr int N = 32 * E;
#pragma unroll
  for (int s = 2; s <= N; s <<= 1) {
#pragma unroll
    for (int d = s >> 1; d > 0; d >>= 1) {
      if (d < E) {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          const int p = j ^ d;
          if (p > j) {
            const bool desc = ((lane * E + j) & s) == 0;
            const V a = v[j], b = v[p];
            const bool swap = desc ? (a < b) : (a > b);
            v[j] = swap ? b : a;
            v[p] = swap ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < E; ++j) {
          V o;
          if constexpr (sizeof(V) == 8) {
            const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v[j]), d / E);
            const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v[j] >> 32), d / E);
            o = (static_cast<V>(hi) << 32) | lo;
          } else {
            o = __shfl_xor_sync(0xFFFFFFFFu, v[j], d / E);
          }
          const int e = lane * E + j;
          const bool keep_max = ((e & d) == 0) == ((e & s) == 0);
          v[j] = keep_max ? (v[j] > o ? v[j] : o) : (v[j] < o ? v[j] : o);
        }
      }
    }
  }
}

// Sorts n <= 32 E winners of cand[] (zero-padded to 32 E) and writes the
// first kk ids to out.
template <int E>
__device__ __forceinline__ void wsel_sort_emit(const uint64_t* cand, int n, int kk,
                                               int32_t* __restrict__ out, int lane) {
  uint64_t x[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int e = lane * E + j;
    x[j] = e < n ? cand[e] : 0ull;
  }
  warp_bitonic_desc<E>(x, lane);
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int r = lane * E + j;
    if (r < kk) out[r] = static_cast<int32_t>(~static_cast<uint32_t>(x[j]));
  }
}

// Inclusive warp scan.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, off);
    if (lane >= off) v += t;
  }
  return v;
}

// The 4 keys at [base, base + 4) of a row in shared memory (16-byte aligned,
// readable up to nb rounded up to 4); bit j of `valid` is set for keys
// below nb.
__device__ __forceinline__ uint4 wsel_ld4(const uint32_t* keys, int base, int nb, uint32_t& valid) {
  if (base >= nb) {
    valid = 0;
    return make_uint4(0u, 0u, 0u, 0u);
  }
  const uint4 v = *reinterpret_cast<const uint4*>(keys + base);
  const int left = nb - base;
  valid = left >= 4 ? 0xFu : ((1u << left) - 1u);
  return v;
}

__device__ __forceinline__ uint32_t wsel_get(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Number of keys of the row >= t (every lane gets it).
__device__ __forceinline__ uint32_t wsel_count_ge(const uint32_t* keys, int nb, uint32_t t, int lane) {
  uint32_t c = 0;
  for (int base = lane * 4; base < nb; base += 128) {
    uint32_t valid;
    const uint4 v = wsel_ld4(keys, base, nb, valid);
#pragma unroll
    for (int j = 0; j < 4; ++j) c += ((valid >> j) & 1u) && wsel_get(v, j) >= t ? 1u : 0u;
  }
  return __reduce_add_sync(0xFFFFFFFFu, c);
}

// Key of a segment maximum; an empty segment (-inf, no key of the row) counts
// as 0, below every score's key.
__device__ __forceinline__ uint32_t base_key_or_zero(float m) {
  return m == -__int_as_float(0x7f800000) ? 0u : score_key(m);
}

// Inverse of score_key for keys of finite scores (the float whose key it is;
// the key of -0.0 and +0.0 maps back to +0.0).
__device__ __forceinline__ float key_to_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Bisection fallback for flat or tied rows (more than kWarpSelCap keys >= T;
// kk < nb): the kk-th largest key value v is found in [T, mx] (count(>= T) >=
// kk, count(>= mx) >= 1); the keys above v are taken with the (kk - #above)
// smallest-index keys equal to v, and the kk winners sorted. keys: the row's
// keys in shared memory.
__device__ __noinline__ void wsel_bisect(const uint32_t* keys, int nb, int kk, uint32_t T, uint32_t mx,
                                         int32_t* __restrict__ out, uint64_t* cand, int lane) {
  uint32_t lo = T, hi = mx;
  while (lo < hi) {
    const uint32_t mid = lo + (hi - lo + 1u) / 2u;
    if (wsel_count_ge(keys, nb, mid, lane) >= static_cast<uint32_t>(kk)) lo = mid;
    else hi = mid - 1u;
  }
  const uint32_t v_k = lo;
  uint32_t above = 0;  // keys above v_k: fewer than kk
  for (int base = lane * 4; base < nb; base += 128) {
    uint32_t valid;
    const uint4 v = wsel_ld4(keys, base, nb, valid);
#pragma unroll
    for (int j = 0; j < 4; ++j) above += ((valid >> j) & 1u) && wsel_get(v, j) > v_k ? 1u : 0u;
  }
  const uint32_t a_incl = warp_incl_scan(above, lane);
  const uint32_t n_above = __shfl_sync(0xFFFFFFFFu, a_incl, 31);
  const uint32_t need = static_cast<uint32_t>(kk) - n_above;
  uint32_t o = a_incl - above;  // this lane's slots for keys above v_k
  uint32_t ties = 0;            // keys equal to v_k before this 128-key block (warp-uniform)
  for (int b0 = 0; b0 < nb; b0 += 128) {
    const int base = b0 + lane * 4;
    uint32_t valid;
    const uint4 v = wsel_ld4(keys, base, nb, valid);
    uint32_t eq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t kv = wsel_get(v, j);
      if ((valid >> j) & 1u) {
        if (kv > v_k) cand[o++] = win_key(kv, base + j);
        eq += kv == v_k ? 1u : 0u;
      }
    }
    // ties in index order: lanes in order, a lane's four keys in order
    const uint32_t e_incl = warp_incl_scan(eq, lane);
    uint32_t r = ties + e_incl - eq;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t kv = wsel_get(v, j);
      if (((valid >> j) & 1u) && kv == v_k) {
        if (r < need) cand[n_above + r] = win_key(kv, base + j);
        ++r;
      }
    }
    ties += __shfl_sync(0xFFFFFFFFu, e_incl, 31);
  }
  __syncwarp();
  wsel_sort_emit<4>(cand, kk, kk, out, lane);
}

// The 4 words at buffer positions [p, p + 4) of a staged row (16-byte
// aligned; p a multiple of 4) whose element i sits at position i + shift;
// bit j of `valid` is set when element p + j - shift lies in [0, nb).
__device__ __forceinline__ uint4 wsel_ld4s(const uint32_t* buf, int p, int shift, int nb, uint32_t& valid) {
  const uint4 v = *reinterpret_cast<const uint4*>(buf + p);
  const int lo = shift - p, hi = nb + shift - p;  // valid j: lo <= j < hi
  valid = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) valid |= (j >= lo && j < hi ? 1u : 0u) << j;
  return v;
}

// Exact top-k (k <= 128) of a row of nb fp32 scores staged in shared memory
// by one warp: element i at buf[i + shift] (0 <= shift < 4, buf 16-byte
// aligned and readable up to nb + shift rounded up to 4; the other words
// there may hold anything). The passes compare the scores as floats against
// the threshold (a float compare orders finite scores as their keys do, -0.0
// == +0.0); only candidates are turned into keys; the bisection fallback
// first moves the row to shift 0 and rewrites it as keys in place. The 128
// segments of the threshold are the buffer positions mod 128. cand:
// kWarpSelCap 64-bit words of this warp's shared memory. Writes out[0, k).
__device__ __forceinline__ void select_row_warp_f32(float* buf, int shift, int nb, int k,
                                                    int32_t* __restrict__ out, uint64_t* cand, int lane) {
  const int kk = k < nb ? k : nb;
  for (int j = kk + lane; j < k; j += 32) out[j] = -1;
  if (kk <= 0) return;
  const uint32_t* bufu = reinterpret_cast<const uint32_t*>(buf);
  const int end = nb + shift;  // buffer positions in use
  float tf = -__int_as_float(0x7f800000);  // -inf: every finite score is a candidate
  uint32_t T = 0, mx = 0;
  if (kk < nb) {
    float m[4] = {tf, tf, tf, tf};  // segment 4 lane + j of {position mod 128}
    for (int p = lane * 4; p < end; p += 128) {
      uint32_t valid;
      const uint4 v = wsel_ld4s(bufu, p, shift, nb, valid);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((valid >> j) & 1u) m[j] = fmaxf(m[j], __uint_as_float(wsel_get(v, j)));
    }
    uint32_t seg[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) seg[j] = base_key_or_zero(m[j]);
    warp_bitonic_desc<4>(seg, lane);
    const int r = kk - 1;
    const uint32_t mine = (r & 3) == 0 ? seg[0] : (r & 3) == 1 ? seg[1] : (r & 3) == 2 ? seg[2] : seg[3];
    mx = __shfl_sync(0xFFFFFFFFu, seg[0], 0);
    T = __shfl_sync(0xFFFFFFFFu, mine, r >> 2);
    tf = key_to_score(T);
  }
  uint32_t c = 0;
  for (int p = lane * 4; p < end; p += 128) {
    uint32_t valid;
    const uint4 v = wsel_ld4s(bufu, p, shift, nb, valid);
#pragma unroll
    for (int j = 0; j < 4; ++j) c += ((valid >> j) & 1u) && __uint_as_float(wsel_get(v, j)) >= tf ? 1u : 0u;
  }
  const uint32_t incl = warp_incl_scan(c, lane);
  const uint32_t n_c = __shfl_sync(0xFFFFFFFFu, incl, 31);
  if (n_c <= static_cast<uint32_t>(kWarpSelCap)) {
    uint32_t o = incl - c;
    for (int p = lane * 4; p < end; p += 128) {
      uint32_t valid;
      const uint4 v = wsel_ld4s(bufu, p, shift, nb, valid);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float x = __uint_as_float(wsel_get(v, j));
        if (((valid >> j) & 1u) && x >= tf) cand[o++] = win_key(score_key(x), p + j - shift);
      }
    }
    __syncwarp();
    if (n_c <= 128u) wsel_sort_emit<4>(cand, static_cast<int>(n_c), kk, out, lane);
    else wsel_sort_emit<8>(cand, static_cast<int>(n_c), kk, out, lane);
    return;
  }
  // Flat or tied rows (kk < nb here): the row moved to shift 0 (chunks of 32
  // in increasing order: each chunk's words are read before they are
  // overwritten, and a write never lands on a word still to be read), then
  // rewritten as keys, then the bisection.
  uint32_t* keys = reinterpret_cast<uint32_t*>(buf);
  for (int i0 = 0; i0 < nb; i0 += 32) {
    const int i = i0 + lane;
    const float x = i < nb ? buf[i + shift] : 0.0f;
    __syncwarp();
    if (i < nb) keys[i] = score_key(x);
    __syncwarp();
  }
  wsel_bisect(keys, nb, kk, T, mx, out, cand, lane);
}

}  // namespace qsa
