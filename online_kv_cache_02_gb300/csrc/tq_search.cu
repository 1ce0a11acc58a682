// Inner-product search over a quantized key database: the decode's two-stage
// estimate of <q, x> for every (query, database vector), without a softmax,
// then the k largest per query.
//
// [P2] "생각정리 209 (TurboQuant)": the method is claimed for KV-cache
// quantization and for vector search (recall against PQ and RabitQ, near-zero
// quantization time); [P4] riverfrot.github.io "TurboQuant란 무엇이며…",
// §4.3: stage-1 reconstruction plus the 1-bit QJL correction is an unbiased
// inner-product estimate.
//
// The database is a K cache of one KV head written by tq_quantize (batch 1,
// n_db tokens): vector t sits in page block_table[t / 16], slot t % 16.
// Three launches: qprep (q~ = Pi q, u = S Pi q, the decode's kernel), the
// scores (CUDA cores: a lane per database vector, eight queries per block,
// codes unpacked from a per-lane copy of the record), and the top k per query
// (radix select of the k-th largest score on its order-preserving bits,
// in-order compaction, bitonic sort by score then index).

#include "tq_internal.h"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

namespace tq {
namespace {

constexpr int kSG = 8;              // queries per scoring block
constexpr int kSThreads = 128;      // four warps, a lane per database vector
constexpr int kSChunk = 2048;       // database vectors per scoring block
constexpr int kSRec = 17;           // words per lane in the staged code records
constexpr int kTThreads = 512;      // top-k block
constexpr int kTMax = 1024;         // largest k
constexpr float kSInvSqrtD = 0.08838834764831845f;
constexpr float kSSqrtHalfPi = 1.2533141373155003f;

struct SearchArgs {
  const float* qprep;        // [nq][d + m]: q~ then u
  int nq, m, n_db, num_pages;
  const uint8_t* kc;
  const int32_t* bt;         // [ceil(n_db / 16)] page ids
  KindLayout kl;
  uint32_t* err;
  float* scores;             // [nq][n_db]
};

// Code of channel j from a vector's code words (the stored format of tq.h).
__device__ __forceinline__ int record_code_at(const unsigned* rec, int bh, int bl, int split, int j) {
  const int grp = j < split ? 0 : 1;
  const int b = grp ? bl : bh;
  const int c = grp ? j - split : j;
  const int base = grp ? split * bh : 0;
  auto bitsat = [&](int off, int n) {
    const unsigned long long pair = (static_cast<unsigned long long>(rec[(off >> 5) + 1]) << 32) | rec[off >> 5];
    return static_cast<int>((pair >> (off & 31)) & ((1u << n) - 1u));
  };
  if (b == 3) {
    const int ob = base + 24 * (c >> 3), i = c & 7;
    if (i < 6) return bitsat(ob + 4 * i, 3);
    const int s = ob + 3 + 4 * (i - 6);
    return bitsat(s, 1) | (bitsat(s + 8, 1) << 1) | (bitsat(s + 16, 1) << 2);
  }
  const int v = bitsat(base + b * c, b);
  if (b == 4) return (v & 8) ? 7 - (v & 7) : 8 + v;
  return v;
}

__global__ void __launch_bounds__(kSThreads) search_score_kernel(SearchArgs s) {
  __shared__ float qt_s[kSG][kD];
  __shared__ float u_s[kSG][kMaxM];
  __shared__ float ck_s[2][16];
  __shared__ unsigned rec_s[kSThreads / 32][32 * kSRec];
  const int q0 = blockIdx.y * kSG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int idx = threadIdx.x; idx < kSG * kD; idx += kSThreads) {
    const int g = idx / kD, j = idx % kD;
    qt_s[g][j] = q0 + g < s.nq ? s.qprep[static_cast<long long>(q0 + g) * (kD + s.m) + j] : 0.0f;
  }
  for (int idx = threadIdx.x; idx < kSG * s.m; idx += kSThreads) {
    const int g = idx / s.m, p = idx % s.m;
    u_s[g][p] = q0 + g < s.nq ? s.qprep[static_cast<long long>(q0 + g) * (kD + s.m) + kD + p] : 0.0f;
  }
  if (threadIdx.x < 32) ck_s[threadIdx.x >> 4][threadIdx.x & 15] = s.kl.g[threadIdx.x >> 4].c[threadIdx.x & 15];
  __syncthreads();

  const long long t0 = static_cast<long long>(blockIdx.x) * kSChunk;
  const long long t1 = min(t0 + kSChunk, static_cast<long long>(s.n_db));
  const int kbh = s.kl.g[0].bits, kbl = s.kl.g[1].bits, ksplit = s.kl.split;
  const int kcw = s.kl.code_bytes / 4;
  const int swords = s.kl.qjl ? s.m / 32 : 0;
  const float qjl_scale = kSSqrtHalfPi / static_cast<float>(s.m);
  unsigned* rec = rec_s[warp] + lane * kSRec;
  for (long long base = t0 + warp * 32; base < t1; base += kSThreads) {
    const long long t = base + lane;
    if (t >= t1) continue;
    const int page = s.bt[t >> 4];
    if (page < 0 || page >= s.num_pages) {      // flagged; the vector cannot rank
      atomicOr(s.err, kErrPage);
      for (int g = 0; g < kSG; ++g)
        if (q0 + g < s.nq) s.scores[static_cast<long long>(q0 + g) * s.n_db + t] = -INFINITY;
      continue;
    }
    const int slot = static_cast<int>(t & 15);
    const unsigned char* kb = s.kc + static_cast<long long>(page) * s.kl.block_bytes;
    const unsigned* cw = reinterpret_cast<const unsigned*>(kb + slot * s.kl.code_bytes);
    for (int w = 0; w < kcw; ++w) rec[w] = cw[w];
    rec[kcw] = 0;
    float s1[kSG], s2[kSG];
#pragma unroll
    for (int g = 0; g < kSG; ++g) s1[g] = s2[g] = 0.0f;
    for (int j = 0; j < kD; ++j) {
      const float c = ck_s[j < ksplit ? 0 : 1][record_code_at(rec, kbh, kbl, ksplit, j)];
#pragma unroll
      for (int g = 0; g < kSG; ++g) s1[g] = fmaf(c, qt_s[g][j], s1[g]);
    }
    const unsigned* sw = reinterpret_cast<const unsigned*>(kb + s.kl.off_signs + slot * (s.m / 8));
    for (int w = 0; w < swords; ++w) {
      const unsigned bits = sw[w];
      for (int i = 0; i < 32; ++i) {
        const bool pos = (bits >> i) & 1u;
#pragma unroll
        for (int g = 0; g < kSG; ++g) s2[g] += pos ? u_s[g][32 * w + i] : -u_s[g][32 * w + i];
      }
    }
    const float nk = __half2float(reinterpret_cast<const __half*>(kb + s.kl.off_norm)[slot]);
    const float rk = s.kl.qjl ? __half2float(reinterpret_cast<const __half*>(kb + s.kl.off_rnorm)[slot]) : 0.0f;
#pragma unroll
    for (int g = 0; g < kSG; ++g)
      if (q0 + g < s.nq)
        s.scores[static_cast<long long>(q0 + g) * s.n_db + t] = fmaf(nk * kSInvSqrtD, s1[g], qjl_scale * rk * s2[g]);
  }
}

// Order-preserving bits of a float: a larger score has a larger key (-0 is
// taken as +0, so equal scores have equal keys).
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix count of `flag` over the block (in thread order) and the
// block's total; every thread must call it.
__device__ __forceinline__ int block_prefix(bool flag, int* warp_tot, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();                                   // warp_tot free from the previous call
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < kTThreads / 32; ++w) {
    const int v = warp_tot[w];
    before += w < warp ? v : 0;
    all += v;
  }
  *total = all;
  return before + in_warp;
}

__global__ void __launch_bounds__(kTThreads) search_topk_kernel(const float* scores, int n, int k, float* top_s,
                                                                 int32_t* top_i) {
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix, s_need;
  __shared__ int warp_tot[kTThreads / 32];
  __shared__ uint32_t out_key[kTMax];
  __shared__ int out_idx[kTMax];
  const int q = blockIdx.x, tid = threadIdx.x;
  const float* sc = scores + static_cast<long long>(q) * n;

  // 1. the key of the k-th largest score, eight bits at a time from the top
  unsigned prefix = 0, mask = 0, need = static_cast<unsigned>(k);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTThreads) {
      const uint32_t key = score_key(sc[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned cum = 0, sel = 0;
      for (int b = 255; b >= 0; --b) {
        if (cum + hist[b] >= need) {
          sel = static_cast<unsigned>(b);
          break;
        }
        cum += hist[b];
      }
      s_prefix = prefix | (sel << shift);
      s_need = need - cum;                 // how many of the keys equal to the prefix so far to take
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
  }
  // prefix is now the k-th largest key; `need` of the scores with that key are taken (lowest indices)
  const int n_gt = k - static_cast<int>(need);

  // 2. in-order compaction: every score above the k-th, then the first `need` equal to it
  for (int i = tid; i < kTMax; i += kTThreads) {
    out_key[i] = 0u;
    out_idx[i] = INT_MAX;
  }
  __syncthreads();
  int base_gt = 0, base_eq = 0;
  for (int tile = 0; tile < n; tile += kTThreads) {
    const int i = tile + tid;
    const uint32_t key = i < n ? score_key(sc[i]) : 0u;
    const bool gt = i < n && key > prefix, eq = i < n && key == prefix;
    int tot_gt, tot_eq;
    const int p_gt = block_prefix(gt, warp_tot, &tot_gt);
    const int p_eq = block_prefix(eq, warp_tot, &tot_eq);
    if (gt) {
      out_key[base_gt + p_gt] = key;
      out_idx[base_gt + p_gt] = i;
    }
    if (eq && base_eq + p_eq < static_cast<int>(need)) {
      out_key[n_gt + base_eq + p_eq] = key;
      out_idx[n_gt + base_eq + p_eq] = i;
    }
    base_gt += tot_gt;
    base_eq += tot_eq;
  }
  __syncthreads();

  // 3. bitonic sort of the kTMax slots: larger key first, equal keys by lower index; the
  // unused slots (key 0, index INT_MAX) sort last
  for (int size = 2; size <= kTMax; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < kTMax; i += kTThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const bool later = out_key[i] < out_key[j] || (out_key[i] == out_key[j] && out_idx[i] > out_idx[j]);
          if (later == up) {
            const uint32_t tk = out_key[i];
            out_key[i] = out_key[j];
            out_key[j] = tk;
            const int ti = out_idx[i];
            out_idx[i] = out_idx[j];
            out_idx[j] = ti;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int r = tid; r < k; r += kTThreads) {
    top_i[static_cast<long long>(q) * k + r] = out_idx[r];
    top_s[static_cast<long long>(q) * k + r] = sc[out_idx[r]];
  }
}

}  // namespace

size_t search_qrows_bytes(int nq, int m) {
  return (sizeof(float) * static_cast<size_t>(nq) * (kD + m) + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_search(const DecodeArgs& qa, const uint8_t* kc, const int32_t* bt, int num_pages, int n_db,
                          int k, float* top_s, int32_t* top_i, float* scores, cudaStream_t st) {
  cudaError_t e = launch_decode(qa, TQ_STAGE_QPREP, st);
  if (e != cudaSuccess) return e;
  SearchArgs s;
  s.qprep = qa.qprep;
  s.nq = qa.B * qa.Hq;
  s.m = qa.m;
  s.n_db = n_db;
  s.num_pages = num_pages;
  s.kc = kc;
  s.bt = bt;
  s.kl = qa.kl;
  s.err = qa.tab.err;
  s.scores = scores;
  const dim3 grid(static_cast<unsigned>((n_db + kSChunk - 1) / kSChunk), static_cast<unsigned>((s.nq + kSG - 1) / kSG));
  search_score_kernel<<<grid, kSThreads, 0, st>>>(s);
  e = cudaGetLastError();
  if (e != cudaSuccess || !top_s) return e;
  search_topk_kernel<<<s.nq, kTThreads, 0, st>>>(s.scores, n_db, k, top_s, top_i);
  return cudaGetLastError();
}

int search_max_k() { return kTMax; }

int search_max_queries() { return 65535 * kSG; }   // the scoring grid's y extent

}  // namespace tq
