// select_row.cuh - exact top-k of one score row by a group of T threads (T a
// multiple of 32, whole warps, synchronised by one named barrier).
//
// Order (Strata pull request 228 part 1 and pull request 856 "Arithmetic
// contract and parity": top-k over the block scores, with a block-index
// tie-break): descending score; equal scores -> smaller block index first;
// -0.0 == +0.0; ids past nb are -1.
//
// Scores are compared as order-preserving uint32 keys (score_key). Rows of
// at most 64 keys are ranked by one warp (select_row_warp64). For k <=
// 128, register-held rows first try a threshold select (select_row_thr: a
// lower bound of the k-th key from per-thread maxima, then an exact rank of
// the few keys above it). Otherwise the search is a radix select on the keys,
// most significant digit first. Register-held rows try a first digit measured down from the row's largest key
// (select_row_window), which nearly always settles the search in one pass;
// otherwise, and for rows in shared memory:
//   * the first digit is fixed, the top 11 key bits (sign, exponent, two
//     mantissa bits: quarter-octave bins);
//   * one suffix scan over the bins finds the digit holding the k-th largest
//     key; every key in a higher bin is a winner;
//   * the search stops as soon as (a) the keys still needed fill the boundary
//     bin exactly, (b) the boundary bin holds at most kSelCandMax keys, which
//     are then ranked by (key, index) directly, or (c) the key is resolved to
//     all 32 bits, when the tied keys with the smallest indices are taken in
//     index order; otherwise the next 8 bits of the boundary bin's keys are
//     histogrammed (a pass over a handful of keys is cheaper than ranking a
//     large bin pairwise);
//   * winners and candidates are gathered by per-thread counts and one group
//     scan (no atomics), and every rank (candidate or final output slot) is
//     computed by several threads per element, reduced with shuffles.
// A winner is the 64-bit key (key << 32 | ~index): all distinct, and larger
// means earlier in the output.
#pragma once

#include "qsa_device.cuh"

namespace qsa {

constexpr int kSelFirstBits = 11;
constexpr int kSelFirstShift = 32 - kSelFirstBits;
constexpr int kSelHistBins = 1 << kSelFirstBits;
constexpr int kSelCandMax = 32;
constexpr int kSelBinMax = 256;
constexpr int kSelRankMax = 32;

struct SelectShared {
  uint32_t wsum[32];
  uint32_t digit, above, cnt;
  uint32_t n_cand;  // window select: candidates gathered so far
};

__device__ __forceinline__ uint32_t lane_mask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <int T>
__device__ __forceinline__ void group_sync(int bar_id) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(T) : "memory");
}

__device__ __forceinline__ uint64_t win_key(uint32_t key, int idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~idx);
}

// Exclusive scan of v over the group in thread order; *total gets the sum.
// Ends with a barrier, so sh.wsum may be reused right after.
template <int T>
__device__ __forceinline__ uint32_t group_excl_scan(uint32_t v, uint32_t* total, SelectShared& sh,
                                                    int gtid, int bar_id) {
  constexpr int kWarps = T / 32;
  const int lane = gtid & 31, gwarp = gtid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sh.wsum[gwarp] = incl;
  group_sync<T>(bar_id);
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t x = sh.wsum[w];
    before += (w < gwarp) ? x : 0u;
    tot += x;
  }
  group_sync<T>(bar_id);
  *total = tot;
  return before + incl - v;
}

// For j < n: emit(j, #{m < n : x[m] > x[j]}). P consecutive threads share an
// element (P a power of two <= 32 with P * n <= T where possible), each
// comparing a strided slice, and add their counts with shuffles.
template <int T, typename Emit>
__device__ __forceinline__ void split_rank(const uint64_t* x, int n, int gtid, Emit emit) {
  int P = 1;
  while (P < 32 && 2 * P * n <= T) P <<= 1;
  const int slots = n * P;
  for (int base = 0; base < slots; base += T) {
    const int t = base + gtid;
    const int e = t / P;
    const int sub = t & (P - 1);
    const bool valid = t < slots;
    const uint64_t me = valid ? x[e] : 0ull;
    uint32_t r = 0;
    if (valid) {
      int m = sub;
#pragma unroll 8
      for (; m < n; m += P) r += x[m] > me ? 1u : 0u;
    }
    for (int o = 1; o < P; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
    if (valid && sub == 0) emit(e, r);
  }
}

// The same ranks over pairs: x is 16-byte aligned and, for odd n, x[n] == 0
// (below every winner key). Thread slot (pair e, sub) compares both elements
// of pair e against the pairs sub, sub + P, ... (one 16-byte load for two
// elements), so a comparison costs half the shared-memory loads of
// split_rank; P is the largest power of two <= 32 with 2 P ceil(n / 2) <= T
// (at least 1).
template <int T, typename Emit>
__device__ __forceinline__ void pair_rank(const uint64_t* x, int n, int gtid, Emit emit) {
  const int np = (n + 1) >> 1;
  int P = 1;
  while (P < 32 && 2 * P * np <= T) P <<= 1;
  const int slots = np * P;
  const ulonglong2* x2 = reinterpret_cast<const ulonglong2*>(x);
  for (int base = 0; base < slots; base += T) {
    const int t = base + gtid;
    const int e = t / P;
    const int sub = t & (P - 1);
    const bool valid = t < slots;
    ulonglong2 me = make_ulonglong2(0ull, 0ull);
    uint32_t r0 = 0, r1 = 0;
    if (valid) {
      me = x2[e];
#pragma unroll 4
      for (int m = sub; m < np; m += P) {
        const ulonglong2 v = x2[m];
        r0 += (v.x > me.x ? 1u : 0u) + (v.y > me.x ? 1u : 0u);
        r1 += (v.x > me.y ? 1u : 0u) + (v.y > me.y ? 1u : 0u);
      }
    }
    for (int o = 1; o < P; o <<= 1) {
      r0 += __shfl_xor_sync(0xFFFFFFFFu, r0, o);
      r1 += __shfl_xor_sync(0xFFFFFFFFu, r1, o);
    }
    if (valid && sub == 0) {
      emit(2 * e, r0);
      if (2 * e + 1 < n) emit(2 * e + 1, r1);
    }
  }
}

// Finds the digit of the bins [0, NBINS) holding the need-th largest key
// (counting from the top bin down); writes digit, count above it and its own
// count to sh. Thread t owns the B = NBINS / T bins [NBINS - (t+1)B, NBINS -
// tB), read with 16-byte loads when B is a multiple of 4.
template <int T, int NBINS>
__device__ __forceinline__ void scan_bins_fixed(const uint32_t* hist, uint32_t need,
                                                SelectShared& sh, int gtid, int bar_id) {
  constexpr int B = NBINS >= T ? NBINS / T : 1;
  const int base = NBINS - (gtid + 1) * B;  // lowest bin of this thread (may be < 0)
  uint32_t c[B];
  if (base >= 0) {
    if constexpr (B % 4 == 0) {
#pragma unroll
      for (int j = 0; j < B; j += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(hist + base + j);
        c[j] = v.x;
        c[j + 1] = v.y;
        c[j + 2] = v.z;
        c[j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < B; ++j) c[j] = hist[base + j];
    }
  } else {
#pragma unroll
    for (int j = 0; j < B; ++j) c[j] = 0;
  }
  uint32_t local = 0;
#pragma unroll
  for (int j = 0; j < B; ++j) local += c[j];
  uint32_t tot;
  const uint32_t excl = group_excl_scan<T>(local, &tot, sh, gtid, bar_id);
  if (excl < need && need <= excl + local) {
    uint32_t run = excl;
    bool found = false;
#pragma unroll
    for (int j = B - 1; j >= 0; --j) {
      if (!found && run + c[j] >= need) {
        sh.digit = static_cast<uint32_t>(base + j);
        sh.above = run;
        sh.cnt = c[j];
        found = true;
      }
      run += c[j];
    }
  }
  group_sync<T>(bar_id);
}

// scan_bins_fixed that also stores, for every bin d, excl[d] = the number of
// keys in the bins above d (thread-owned bins, 16-byte stores).
template <int T, int NBINS>
__device__ __forceinline__ void scan_bins_excl(const uint32_t* hist, uint32_t* excl, uint32_t need,
                                               SelectShared& sh, int gtid, int bar_id) {
  static_assert(NBINS % T == 0 && (NBINS / T) % 4 == 0, "whole 16-byte groups per thread");
  constexpr int B = NBINS / T;
  const int base = NBINS - (gtid + 1) * B;
  uint32_t c[B];
#pragma unroll
  for (int j = 0; j < B; j += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(hist + base + j);
    c[j] = v.x;
    c[j + 1] = v.y;
    c[j + 2] = v.z;
    c[j + 3] = v.w;
  }
  uint32_t local = 0;
#pragma unroll
  for (int j = 0; j < B; ++j) local += c[j];
  uint32_t tot;
  const uint32_t ex = group_excl_scan<T>(local, &tot, sh, gtid, bar_id);
  uint32_t e[B];
  uint32_t run = ex;
#pragma unroll
  for (int j = B - 1; j >= 0; --j) {
    e[j] = run;
    if (run < need && need <= run + c[j]) {
      sh.digit = static_cast<uint32_t>(base + j);
      sh.above = run;
      sh.cnt = c[j];
    }
    run += c[j];
  }
#pragma unroll
  for (int j = 0; j < B; j += 4)
    *reinterpret_cast<uint4*>(excl + base + j) = make_uint4(e[j], e[j + 1], e[j + 2], e[j + 3]);
  group_sync<T>(bar_id);
}

// The same for a run-time number of bins (2048 or 256).
template <int T>
__device__ __forceinline__ void scan_bins(const uint32_t* hist, int nbins, uint32_t need,
                                          SelectShared& sh, int gtid, int bar_id) {
  if (nbins == kSelHistBins) scan_bins_fixed<T, kSelHistBins>(hist, need, sh, gtid, bar_id);
  else scan_bins_fixed<T, 256>(hist, need, sh, gtid, bar_id);
}

// ------------------------------------------------- register-resident keys
// Thread gtid holds the keys of indices j*T + gtid, j < R (key 0 past nb: it
// is below every finite score's key). Fewer instructions per element than
// the shared-memory path, for rows with nb <= R*T.

// Top-k of one row whose keys are in registers and whose first-digit
// histogram is complete in hist (build_first_digit_hist below).
template <int T, int R>
__device__ void select_row_regs(const uint32_t (&key)[R], int nb, int k, int32_t* __restrict__ out,
                                uint32_t* hist, uint64_t* cand, uint64_t* sel, SelectShared& sh,
                                int gtid, int bar_id) {
  const int kk = k < nb ? k : nb;
  enum Mode { kTakeAll, kTies, kCand };
  Mode mode = kTakeAll;
  uint32_t thr = 0;
  uint32_t need = static_cast<uint32_t>(kk);
  uint32_t prefix = 0;
  int hi = 32;
  if (kk > 0 && kk < nb) {
    int nbits = kSelFirstBits;
    bool first = true;
    while (true) {
      const int lo = hi - nbits;
      const int nbins = 1 << nbits;
      if (!first) {
        const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
        for (int i = gtid; i < 256; i += T) hist[i] = 0;  // refinement scans read 256 bins
        group_sync<T>(bar_id);
#pragma unroll
        for (int j = 0; j < R; ++j) {
          if (j * T + gtid < nb && ((key[j] ^ prefix) >> hi) == 0)
            atomicAdd(&hist[(key[j] >> lo) & dmask], 1u);
        }
        group_sync<T>(bar_id);
      }
      first = false;
      scan_bins<T>(hist, nbins, need, sh, gtid, bar_id);
      const uint32_t digit = sh.digit, above = sh.above, cnt = sh.cnt;
      need -= above;
      prefix |= digit << lo;
      hi = lo;
      if (cnt == need) {
        mode = kTakeAll;
        thr = prefix;
        break;
      }
      if (hi == 0) {
        mode = kTies;
        thr = prefix;
        break;
      }
      if (cnt <= static_cast<uint32_t>(kSelCandMax)) {
        mode = kCand;
        break;
      }
      nbits = hi < 8 ? hi : 8;
      group_sync<T>(bar_id);
    }
  }

  if (kk > 0) {
    // Winner / candidate flags per register key (key 0 never qualifies).
    uint32_t wmask = 0, cmask = 0;
    if (mode == kCand) {
      const uint32_t bin_top = prefix | ((1u << hi) - 1u);
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const bool valid = j * T + gtid < nb;
        const bool w = valid && key[j] > bin_top;
        const bool c = valid && !w && ((key[j] ^ prefix) >> hi) == 0;
        wmask |= (w ? 1u : 0u) << j;
        cmask |= (c ? 1u : 0u) << j;
      }
    } else {
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const bool valid = j * T + gtid < nb;
        const bool w = valid && (mode == kTakeAll ? key[j] >= thr : key[j] > thr);
        wmask |= (w ? 1u : 0u) << j;
      }
    }
    uint32_t totals;
    const uint32_t offs = group_excl_scan<T>((static_cast<uint32_t>(__popc(wmask)) << 16) |
                                                 static_cast<uint32_t>(__popc(cmask)),
                                             &totals, sh, gtid, bar_id);
    uint32_t wo = offs >> 16, co = offs & 0xFFFFu;
    const uint32_t n_win = totals >> 16, n_cand = totals & 0xFFFFu;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (wmask & (1u << j)) sel[wo++] = win_key(key[j], j * T + gtid);
      if (cmask & (1u << j)) cand[co++] = win_key(key[j], j * T + gtid);
    }
    group_sync<T>(bar_id);
    if (mode == kCand) {
      const uint32_t nd = need;
      split_rank<T>(cand, static_cast<int>(n_cand), gtid, [&](int e, uint32_t r) {
        if (r < nd) sel[n_win + r] = cand[e];
      });
      group_sync<T>(bar_id);
    } else if (mode == kTies) {
      uint32_t taken = 0;  // uniform over the group; slices j in index order
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (taken >= need) break;
        const int i = j * T + gtid;
        const bool tie = i < nb && key[j] == thr;
        uint32_t tot;
        const uint32_t r = taken + group_excl_scan<T>(tie ? 1u : 0u, &tot, sh, gtid, bar_id);
        if (tie && r < need) sel[n_win + r] = win_key(thr, i);
        taken += tot;
      }
      group_sync<T>(bar_id);
    }
  }

  // Output slot of every winner: its rank among the winners.
  split_rank<T>(sel, kk, gtid, [&](int e, uint32_t r) {
    out[r] = static_cast<int32_t>(~static_cast<uint32_t>(sel[e]));
  });
  for (int j = kk + gtid; j < k; j += T) out[j] = -1;
}

// ------------------------------------------------ window select (registers)
// The same search with a first digit measured down from the row's largest
// key M: digit kSelHistBins-1-b holds the keys with (M - key) >> kSelWinShift
// == b, for b < kSelHistBins - 1 (the 32 octaves of fp32 below M in steps of
// 1/64 octave, wide enough to reach past a +1e9 tail score); keys further
// below get digit 0 and are not counted. Score rows are dense near their
// top, so the k-th largest key nearly always lies in the window, in a bin of
// a few keys: one histogram and one scan finish the search. The scan also
// leaves each bin's output offset (the keys in higher bins), so winners are
// scattered straight to their bin's slots and ordered inside the bin, and
// the boundary bin's keys are ranked directly. Otherwise
// (the k-th key below the window, or more than kSelBinMax keys in its bin)
// the function returns false having written only hist and sh, and the
// caller runs the fixed-digit select (select_row_regs). hist must be zero on
// entry; excl holds kSelHistBins words (16-byte aligned), sel_bin k words;
// keys past nb are 0.
constexpr int kSelWinShift = 17;

// Loads keys already in shared memory into registers and zeroes hist (the
// first barrier of select_row_window orders the zeroing).
template <int T, int R>
__device__ __forceinline__ void load_keys_regs(const uint32_t* keys, int nb, uint32_t (&key)[R],
                                               uint32_t* hist, int gtid) {
  for (int i = gtid * 4; i < kSelHistBins; i += T * 4)
    *reinterpret_cast<uint4*>(hist + i) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = j * T + gtid;
    key[j] = i < nb ? keys[i] : 0u;
  }
}

// The same from a row of scores in global memory (ld.global.cg).
template <int T, int R>
__device__ __forceinline__ void load_keys_regs_global(const float* s, int nb, uint32_t (&key)[R],
                                                      uint32_t* hist, int gtid) {
  float v[R];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int i = j * T + gtid;
    v[j] = i < nb ? __ldcg(s + i) : 0.0f;
  }
  for (int i = gtid * 4; i < kSelHistBins; i += T * 4)
    *reinterpret_cast<uint4*>(hist + i) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int j = 0; j < R; ++j) key[j] = j * T + gtid < nb ? score_key(v[j]) : 0u;
}

// Rebuilds hist as the fixed first-digit histogram of register keys (the
// entry state of select_row_regs).
template <int T, int R>
__device__ __forceinline__ void build_first_digit_hist(const uint32_t (&key)[R], int nb,
                                                       uint32_t* hist, int gtid, int bar_id) {
  for (int i = gtid * 4; i < kSelHistBins; i += T * 4)
    *reinterpret_cast<uint4*>(hist + i) = make_uint4(0u, 0u, 0u, 0u);
  group_sync<T>(bar_id);
#pragma unroll
  for (int j = 0; j < R; ++j)
    if (j * T + gtid < nb) atomicAdd(&hist[key[j] >> kSelFirstShift], 1u);
  group_sync<T>(bar_id);
}

template <int T, int R>
__device__ bool select_row_window(const uint32_t (&key)[R], int nb, int k,
                                  int32_t* __restrict__ out, uint32_t* hist, uint32_t* excl,
                                  uint64_t* cand, uint64_t* sel, uint32_t* sel_bin,
                                  SelectShared& sh, int gtid, int bar_id) {
  constexpr int kWarps = T / 32;
  constexpr uint32_t kTop = kSelHistBins - 1;
  const int kk = k < nb ? k : nb;
  if (kk < nb) {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < R; ++j) m = max(m, key[j]);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((gtid & 31) == 0) sh.wsum[gtid >> 5] = m;
    if (gtid == 0) {
      sh.cnt = 0xFFFFFFFFu;  // stays so unless the scan finds the digit
      sh.n_cand = 0;
    }
    group_sync<T>(bar_id);
    uint32_t M = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = max(M, sh.wsum[w]);
    auto digit = [&](uint32_t kv) {
      const uint32_t t = (M - kv) >> kSelWinShift;
      return t < kTop ? kTop - t : 0u;
    };
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t d = digit(key[j]);
      if (j * T + gtid < nb && d > 0) atomicAdd(&hist[d], 1u);
    }
    group_sync<T>(bar_id);
    scan_bins_excl<T, kSelHistBins>(hist, excl, static_cast<uint32_t>(kk), sh, gtid, bar_id);
    const uint32_t cnt = sh.cnt;
    if (cnt == 0xFFFFFFFFu) return false;  // the k-th key lies below the window
    const uint32_t bdig = sh.digit, above = sh.above;
    const uint32_t need = static_cast<uint32_t>(kk) - above;
    const bool take_bin = cnt == need;
    if (!take_bin && cnt > static_cast<uint32_t>(kSelBinMax)) return false;

    // Winners (digits above the boundary, and the boundary bin when it is
    // taken whole) go to a slot in their bin's output range [excl[d],
    // excl[d-1]) (the boundary digit is at least 1: digit 0 is not counted);
    // otherwise the boundary bin's keys become candidates.
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t d = digit(key[j]);
      if (j * T + gtid < nb && d >= bdig) {
        const uint64_t wk = win_key(key[j], j * T + gtid);
        if (d > bdig || take_bin) {
          const uint32_t slot = excl[d] + atomicSub(&hist[d], 1u) - 1u;
          sel[slot] = wk;
          sel_bin[slot] = d;
        } else {
          cand[atomicAdd(&sh.n_cand, 1u)] = wk;
        }
      }
    }
    group_sync<T>(bar_id);
    // Order inside each winner's bin (bins hold a few keys), P threads per
    // winner, and the candidates' ranks: every output slot is written once.
    const int n_win = static_cast<int>(take_bin ? static_cast<uint32_t>(kk) : above);
    int P = 1;
    while (P < 32 && 2 * P * n_win <= T) P <<= 1;
    for (int b0 = 0; b0 < n_win * P; b0 += T) {
      const int t = b0 + gtid, e = t / P, sub = t & (P - 1);
      const bool valid = e < n_win;
      uint64_t me = 0;
      uint32_t lo = 0, r = 0;
      if (valid) {
        me = sel[e];
        const uint32_t d = sel_bin[e];
        lo = excl[d];
        const uint32_t hi = excl[d - 1];
        for (uint32_t i = lo + sub; i < hi; i += P) r += sel[i] > me ? 1u : 0u;
      }
      for (int o = 1; o < P; o <<= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, o);
      if (valid && sub == 0) out[lo + r] = static_cast<int32_t>(~static_cast<uint32_t>(me));
    }
    if (!take_bin) {
      const int n_c = static_cast<int>(cnt);
      for (int e = gtid; e < n_c; e += T) {
        const uint64_t me = cand[e];
        uint32_t r = 0;
        for (int i = 0; i < n_c; ++i) r += cand[i] > me ? 1u : 0u;
        if (r < need) out[above + r] = static_cast<int32_t>(~static_cast<uint32_t>(me));
      }
    }
    return true;
  }

  // kk == nb: every key is a winner (and ids past nb are -1).
  uint32_t wmask = 0;
#pragma unroll
  for (int j = 0; j < R; ++j) wmask |= (j * T + gtid < nb ? 1u : 0u) << j;
  uint32_t n_win;
  uint32_t wo = group_excl_scan<T>(static_cast<uint32_t>(__popc(wmask)), &n_win, sh, gtid, bar_id);
#pragma unroll
  for (int j = 0; j < R; ++j)
    if (wmask & (1u << j)) sel[wo++] = win_key(key[j], j * T + gtid);
  group_sync<T>(bar_id);
  split_rank<T>(sel, kk, gtid, [&](int e, uint32_t r) {
    out[r] = static_cast<int32_t>(~static_cast<uint32_t>(sel[e]));
  });
  for (int j = kk + gtid; j < k; j += T) out[j] = -1;
  return true;
}

// ------------------------------------------ one warp, rows of <= 64 keys
// Short rows (nb <= 64): lane l holds the keys of indices l and l + 32 (any
// value past nb: those entries never count), and every key is ranked against
// the others by (key, index) with shuffles; ranks below k are the output
// slots and slots past nb get -1. No block barrier: the rest of the group
// may idle.
__device__ __forceinline__ void select_row_warp64(uint32_t key0, uint32_t key1, int nb, int k,
                                                  int32_t* __restrict__ out, int lane) {
  const bool v0 = lane < nb, v1 = lane + 32 < nb;
  // A winner key is never 0 (its low word is ~index), so 0 marks an empty entry.
  const uint64_t w0 = v0 ? win_key(key0, lane) : 0ull;
  const uint64_t w1 = v1 ? win_key(key1, lane + 32) : 0ull;
  uint32_t r0 = 0, r1 = 0;
#pragma unroll 8
  for (int s = 0; s < 32; ++s) {
    const uint64_t y0 = __shfl_sync(0xFFFFFFFFu, w0, s);
    const uint64_t y1 = __shfl_sync(0xFFFFFFFFu, w1, s);
    r0 += (y0 > w0 ? 1u : 0u) + (y1 > w0 ? 1u : 0u);
    r1 += (y0 > w1 ? 1u : 0u) + (y1 > w1 ? 1u : 0u);
  }
  if (v0 && r0 < static_cast<uint32_t>(k)) out[r0] = lane;
  if (v1 && r1 < static_cast<uint32_t>(k)) out[r1] = lane + 32;
  for (int j = nb + lane; j < k; j += 32) out[j] = -1;
}

// ------------------------------------------- threshold select (registers)
// For k <= kSelThrKMax and k < nb: a lower bound T of the k-th largest key
// from per-thread maxima, then an exact rank of the few keys >= T.
//   * each thread's R keys form a segment; warp w takes t_w, the q-th
//     largest of its 32 segment maxima (q = ceil(k / warps)), by q rounds of
//     a warp max with the round's maxima removed (equal maxima leave together,
//     which can only lower t_w). At least q keys of warp w are >= t_w, so at
//     least k keys of the row are >= T = min_w t_w: every winner is >= T.
//   * the keys >= T (about 1.5-2 k on score rows) are gathered in thread
//     order (a warp scan, then the warps' totals), and each is ranked among
//     them by (key, index) (pair_rank); ranks below k are the output slots.
// Three group barriers in all. Returns false, after a barrier and having
// written nothing but cand and sh, when more than kSelBinMax keys are >= T
// (ties or flat rows), or when k >= nb or k > kSelThrKMax; the caller then
// runs the window select (hist must still be zero for it). cand must be
// 16-byte aligned.
// Measured against the window select on the same rows (one 256-thread CTA
// per row, three per SM): 3,856 vs 4,297 cycles per 2048-key row, 2,646 vs
// 3,800 per 513-key row. Gathering into per-warp slots, or ranking with warp
// sums, or sorting the candidates with one warp's bitonic network were each
// slower (4,365 / 5,557 cycles): shuffles and warp reductions are the scarce
// resource when several CTAs share an SM. The gather by the warps' totals
// instead of one shared counter, and the ranking over pairs instead of
// single elements, took a 2048-key row from 3,314 to 3,126 cycles (one CTA
// per SM) and from 4,038 to 3,795 (one CTA per row).
constexpr int kSelThrKMax = 128;

template <int T, int R>
__device__ bool select_row_thr(const uint32_t (&key)[R], int nb, int k, int32_t* __restrict__ out,
                               uint64_t* cand, SelectShared& sh, int gtid, int bar_id) {
  constexpr int kWarps = T / 32;
  static_assert(2 * kWarps <= 32, "sh.wsum holds the warps' thresholds and totals");
  if (k >= nb || k > kSelThrKMax) return false;
  const int lane = gtid & 31, warp = gtid >> 5;
  const int q = (k + kWarps - 1) / kWarps;
  uint32_t m = 0;  // keys past nb are 0, below every score's key
#pragma unroll
  for (int j = 0; j < R; ++j) m = max(m, key[j]);
  uint32_t v = m, t = 0;
  for (int i = 0; i < q; ++i) {
    t = __reduce_max_sync(0xFFFFFFFFu, v);
    if (v == t) v = 0;
  }
  if (lane == 0) sh.wsum[warp] = t;
  group_sync<T>(bar_id);
  uint32_t thr = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) thr = min(thr, sh.wsum[w]);
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < R; ++j) c += (j * T + gtid < nb && key[j] >= thr) ? 1u : 0u;
  uint32_t incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) sh.wsum[kWarps + warp] = incl;
  group_sync<T>(bar_id);
  uint32_t o = incl - c, n_c = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t x = sh.wsum[kWarps + w];
    o += w < warp ? x : 0u;
    n_c += x;
  }
#pragma unroll
  for (int j = 0; j < R; ++j) {
    if (j * T + gtid < nb && key[j] >= thr) {
      if (o < static_cast<uint32_t>(kSelBinMax)) cand[o] = win_key(key[j], j * T + gtid);
      ++o;
    }
  }
  // pair_rank reads cand[n_c] for odd n_c: a zero key ranks below them all.
  if (gtid == 0 && (n_c & 1u) && n_c < static_cast<uint32_t>(kSelBinMax)) cand[n_c] = 0ull;
  group_sync<T>(bar_id);
  if (n_c > static_cast<uint32_t>(kSelBinMax)) {
    group_sync<T>(bar_id);  // every thread is past its reads of sh before it is reused
    return false;
  }
  pair_rank<T>(cand, static_cast<int>(n_c), gtid, [&](int e, uint32_t r) {
    if (r < static_cast<uint32_t>(k)) out[r] = static_cast<int32_t>(~static_cast<uint32_t>(cand[e]));
  });
  return true;
}

// ------------------------------------------------ G-warp select, keys in smem
// A group of G warps (T = 32 G threads) selects one row whose keys are in
// shared memory. Per-element work is a histogram increment and two compares;
// everything else is a fixed cost per warp, which is why a row gets only a
// few warps. After the first 11-bit digit, the boundary bin's keys (at most
// kSelBinMax of them) are compacted and only they are refined, 8 bits at a
// time, until the keys still needed fill a bin or at most kSelRankMax remain,
// which are ranked pairwise.

struct GroupShared {
  uint32_t wsum[8];
  uint32_t digit, above, cnt, seg;
};

// Exclusive scan over the group; ends with a barrier (wsum reusable after).
template <int T>
__device__ __forceinline__ uint32_t gscan(uint32_t v, uint32_t* total, GroupShared& sh, int gtid,
                                          int bar_id) {
  constexpr int W = T / 32;
  const int lane = gtid & 31, gw = gtid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += t;
  }
  if (W == 1) {
    *total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    __syncwarp();
    return incl - v;
  }
  if (lane == 31) sh.wsum[gw] = incl;
  group_sync<T>(bar_id);
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const uint32_t x = sh.wsum[w];
    before += (w < gw) ? x : 0u;
    tot += x;
  }
  group_sync<T>(bar_id);
  *total = tot;
  return before + incl - v;
}

// Boundary digit among NB bins: the bin holding the need-th largest key.
// Thread t owns bins [NB - (t+1)B, NB - tB) with B = NB / T (>= 1); the owner
// of the boundary hands its B bins to warp 0, which finds the bin with one
// more warp scan. Result in sh (digit, above, cnt), after a barrier.
template <int T, int NB>
__device__ __forceinline__ void gfind(const uint32_t* hist, uint32_t need, GroupShared& sh,
                                      int gtid, int bar_id) {
  constexpr int B = NB >= T ? NB / T : 1;
  const int lane = gtid & 31;
  const int base = NB - (gtid + 1) * B;
  uint32_t local = 0;
  if (base >= 0) {
    if constexpr (B % 4 == 0) {
      // rotated 16-byte reads: lanes start at different 16-byte units
#pragma unroll
      for (int c = 0; c < B / 4; ++c) {
        const int u = (c + lane) % (B / 4);
        const uint4 v = *reinterpret_cast<const uint4*>(hist + base + 4 * u);
        local += v.x + v.y + v.z + v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < B; ++j) local += hist[base + j];
    }
  }
  uint32_t tot;
  const uint32_t excl = gscan<T>(local, &tot, sh, gtid, bar_id);
  if (excl < need && need <= excl + local) {
    sh.seg = static_cast<uint32_t>(gtid);
    sh.above = excl;  // count above this thread's segment
  }
  group_sync<T>(bar_id);
  if (gtid < 32) {
    // Warp 0: the B bins of the boundary segment, one or more per lane, top first.
    const int sbase = NB - (static_cast<int>(sh.seg) + 1) * B;
    const uint32_t above0 = sh.above;
    constexpr int PER = B >= 32 ? B / 32 : 1;
    uint32_t c[PER];
    uint32_t lsum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int bin = sbase + B - 1 - (lane * PER + j);  // lane 0 holds the top bins
      c[j] = (lane * PER + j < B) ? hist[bin] : 0u;
      lsum += c[j];
    }
    uint32_t incl = lsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += t;
    }
    const uint32_t ex = above0 + incl - lsum;
    if (ex < need && need <= ex + lsum) {
      uint32_t run = ex;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        if (run < need && need <= run + c[j]) {
          sh.digit = static_cast<uint32_t>(sbase + B - 1 - (lane * PER + j));
          sh.above = run;
          sh.cnt = c[j];
        }
        run += c[j];
      }
    }
  }
  group_sync<T>(bar_id);
}

// Top-k of a row whose keys[0..nb) are in shared memory (visible to the
// group). hist: kSelHistBins words, 16-byte aligned; cand: kSelBinMax;
// sel: min(k, nb). Writes out[0..k).
template <int G>
__device__ void select_row_g(const uint32_t* keys, int nb, int k, int32_t* __restrict__ out,
                             uint32_t* hist, uint64_t* cand, uint64_t* sel, GroupShared& sh,
                             int gtid, int bar_id) {
  constexpr int T = 32 * G;
  const int kk = k < nb ? k : nb;
  enum Mode { kTakeAll, kTies, kCandidates };
  Mode mode = kTakeAll;
  uint32_t thr = 0, need = static_cast<uint32_t>(kk), prefix = 0;
  int hi = 32;
  uint32_t n_cand = 0;

  if (kk > 0 && kk < nb) {
    // ---- first digit over all keys
    for (int i = gtid * 4; i < kSelHistBins; i += 4 * T)
      *reinterpret_cast<uint4*>(hist + i) = make_uint4(0u, 0u, 0u, 0u);
    group_sync<T>(bar_id);
#pragma unroll 8
    for (int i = gtid; i < nb; i += T) atomicAdd(&hist[keys[i] >> kSelFirstShift], 1u);
    group_sync<T>(bar_id);
    gfind<T, kSelHistBins>(hist, need, sh, gtid, bar_id);
    {
      const uint32_t digit = sh.digit, cnt = sh.cnt;
      need -= sh.above;
      prefix = digit << kSelFirstShift;
      hi = kSelFirstShift;
      if (cnt == need) {
        mode = kTakeAll;
        thr = prefix;
      } else {
        mode = kCandidates;
        n_cand = cnt;
      }
    }
    // ---- full 8-bit passes while the boundary bin is too large to compact
    while (mode == kCandidates && n_cand > static_cast<uint32_t>(kSelBinMax)) {
      const int nbits = hi < 8 ? hi : 8;
      const int lo = hi - nbits;
      const uint32_t dmask = (1u << nbits) - 1u;
      group_sync<T>(bar_id);
      for (int i = gtid; i < 256; i += T) hist[i] = 0;
      group_sync<T>(bar_id);
#pragma unroll 8
      for (int i = gtid; i < nb; i += T) {
        const uint32_t key = keys[i];
        if (((key ^ prefix) >> hi) == 0) atomicAdd(&hist[(key >> lo) & dmask], 1u);
      }
      group_sync<T>(bar_id);
      gfind<T, 256>(hist, need, sh, gtid, bar_id);
      const uint32_t digit = sh.digit, cnt = sh.cnt;
      need -= sh.above;
      prefix |= digit << lo;
      hi = lo;
      if (cnt == need) {
        mode = kTakeAll;
        thr = prefix;
      } else if (hi == 0) {
        mode = kTies;
        thr = prefix;
      } else {
        n_cand = cnt;
      }
    }
  }

  uint32_t n_win = 0;
  if (kk > 0) {
    // ---- gather: count, scan, write (winners -> sel, boundary keys -> cand)
    const uint32_t bin_top = (mode == kCandidates) ? (prefix | ((1u << hi) - 1u)) : 0u;
    uint32_t cw = 0, cc = 0;
#pragma unroll 8
    for (int i = gtid; i < nb; i += T) {
      const uint32_t key = keys[i];
      if (mode == kTakeAll) {
        cw += key >= thr ? 1u : 0u;
      } else if (mode == kTies) {
        cw += key > thr ? 1u : 0u;
      } else {
        const bool w = key > bin_top;
        cw += w ? 1u : 0u;
        cc += (!w && ((key ^ prefix) >> hi) == 0) ? 1u : 0u;
      }
    }
    uint32_t totals;
    const uint32_t offs = gscan<T>((cw << 16) | cc, &totals, sh, gtid, bar_id);
    uint32_t wo = offs >> 16, co = offs & 0xFFFFu;
    n_win = totals >> 16;
    if (cw | cc) {
#pragma unroll 8
      for (int i = gtid; i < nb; i += T) {
        const uint32_t key = keys[i];
        bool w, c = false;
        if (mode == kTakeAll) {
          w = key >= thr;
        } else if (mode == kTies) {
          w = key > thr;
        } else {
          w = key > bin_top;
          c = !w && ((key ^ prefix) >> hi) == 0;
        }
        if (w) sel[wo++] = win_key(key, i);
        if (c) cand[co++] = win_key(key, i);
      }
    }
    group_sync<T>(bar_id);

    if (mode == kCandidates) {
      // ---- refine the compacted boundary keys, 8 bits at a time
      while (n_cand > static_cast<uint32_t>(kSelRankMax) && hi > 0) {
        const int nbits = hi < 8 ? hi : 8;
        const int lo = hi - nbits;
        for (int i = gtid; i < 256; i += T) hist[i] = 0;
        group_sync<T>(bar_id);
        for (int c = gtid; c < static_cast<int>(n_cand); c += T)
          atomicAdd(&hist[(static_cast<uint32_t>(cand[c] >> 32) >> lo) & ((1u << nbits) - 1u)], 1u);
        group_sync<T>(bar_id);
        gfind<T, 256>(hist, need, sh, gtid, bar_id);
        const uint32_t digit = sh.digit, cnt = sh.cnt;
        const uint32_t above = sh.above;
        const uint32_t new_prefix = prefix | (digit << lo);
        // candidates above the new bin are winners; those in it stay
        constexpr int kPer = (kSelBinMax + T - 1) / T;
        uint32_t fw = 0, fc = 0;
        uint64_t mine[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int c = gtid + j * T;
          mine[j] = c < static_cast<int>(n_cand) ? cand[c] : 0ull;
          const uint32_t d = (static_cast<uint32_t>(mine[j] >> 32) >> lo) & ((1u << nbits) - 1u);
          fw += (c < static_cast<int>(n_cand) && d > digit) ? 1u : 0u;
          fc += (c < static_cast<int>(n_cand) && d == digit) ? 1u : 0u;
        }
        uint32_t tt;
        const uint32_t o = gscan<T>((fw << 16) | fc, &tt, sh, gtid, bar_id);  // cand reads done
        uint32_t wo2 = n_win + (o >> 16), co2 = o & 0xFFFFu;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          const int c = gtid + j * T;
          const uint32_t d = (static_cast<uint32_t>(mine[j] >> 32) >> lo) & ((1u << nbits) - 1u);
          if (c < static_cast<int>(n_cand)) {
            if (d > digit) sel[wo2++] = mine[j];
            else if (d == digit) cand[co2++] = mine[j];
          }
        }
        group_sync<T>(bar_id);
        n_win += tt >> 16;
        need -= above;
        prefix = new_prefix;
        hi = lo;
        n_cand = cnt;
        if (cnt == need) {
          // every key left in the bin is a winner
          for (int c = gtid; c < static_cast<int>(cnt); c += T) sel[n_win + c] = cand[c];
          group_sync<T>(bar_id);
          n_win += cnt;
          need = 0;
          n_cand = 0;
          break;
        }
      }
      // ---- rank the last candidates pairwise; the top `need` are winners
      const uint32_t nd = need, nw = n_win;
      split_rank<T>(cand, static_cast<int>(n_cand), gtid, [&](int e, uint32_t r) {
        if (r < nd) sel[nw + r] = cand[e];
      });
      group_sync<T>(bar_id);
    } else if (mode == kTies) {
      uint32_t taken = 0;
      for (int base = 0; base < nb && taken < need; base += T) {
        const int i = base + gtid;
        const bool tie = i < nb && keys[i] == thr;
        uint32_t tot;
        const uint32_t r = taken + gscan<T>(tie ? 1u : 0u, &tot, sh, gtid, bar_id);
        if (tie && r < need) sel[n_win + r] = win_key(thr, i);
        taken += tot;
      }
      group_sync<T>(bar_id);
    }
  }

  // ---- output slot of every winner: its rank among the winners
  split_rank<T>(sel, kk, gtid, [&](int e, uint32_t r) {
    out[r] = static_cast<int32_t>(~static_cast<uint32_t>(sel[e]));
  });
  for (int j = kk + gtid; j < k; j += T) out[j] = -1;
}


}  // namespace qsa
