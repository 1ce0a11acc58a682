// Decode attention over the packed, paged cache.
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.2-§2.3 (decode: the new
// token's query against every cached key, softmax, weighted sum of values),
// §4.3 (stage-1 reconstruction plus the QJL 1-bit correction gives an unbiased
// inner product; softmax(Q K^T / sqrt(d))); [P2] "생각정리 209 (TurboQuant)",
// stage 2 (the residual's 1-bit sketch makes the inner product unbiased).
//
// Three launches on one stream:
//   qprep  : q~ = Pi q, u = S q~ = (S Pi) q (fp32) per query head
//   chunk  : per (chunk, KV head, sequence): every cached key t of the chunk is
//            scored as (n_t/sqrt(d)) <q~, c[code_t]> + sqrt(pi/2)/m rho_t
//            <u, +-1_t>, an online (flash-style) softmax keeps (max, sum,
//            acc[d]) per query head, acc += p_t (nv_t/sqrt(d)) c_v[code_t]
//   merge  : log-sum-exp merge of the chunk partials, o = Pi^T (acc / sum)
// The G query heads that share a KV head share every unpacked key and value.

#include "tq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace tq {
namespace {

constexpr int kThreads = 128;
constexpr int kRecStride = 17;     // words per lane in the staged key-code records
constexpr float kInvSqrtD = 0.08838834764831845f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;   // sqrt(pi/2)

__device__ __forceinline__ float load_q(const void* q, bool f32, long long idx) {
  if (f32) return static_cast<const float*>(q)[idx];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(q)[idx]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// [q~; u] = W q with W = [Pi; S Pi] (fp32, built once at create time): a
// block takes 32 query heads x 64 outputs; its 32 KB slice of W^T arrives in
// one round of independent 16-byte loads (dynamic shared memory), then four
// groups of 128 threads take a quarter of k each, a thread a 4 heads x 4
// outputs tile (one 16-byte W load and four broadcast q loads per 16 FMAs);
// the four partial tiles are summed through shared memory.
constexpr int kQP = 32;
constexpr int kQO = 64;
constexpr int kQThreads = 512;
constexpr int kQK = kD / (kQThreads / 128);      // k per group
constexpr int kQPad = kD + 4;                   // q rows, padded
constexpr int kQprepSmem = (kD * kQO + kQP * kQPad + (kQThreads / 128) * kQP * kQO) * 4;

__global__ void __launch_bounds__(kQThreads) qprep_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float qsm[];
  float(*ws)[kQO] = reinterpret_cast<float(*)[kQO]>(qsm);
  float(*qs)[kQPad] = reinterpret_cast<float(*)[kQPad]>(qsm + kD * kQO);
  float(*ps)[kQP][kQO] = reinterpret_cast<float(*)[kQP][kQO]>(qsm + kD * kQO + kQP * kQPad);   // partial tiles
  const int nout = kD + a.m;
  const long long r0 = static_cast<long long>(blockIdx.x) * kQP;
  const int c0 = blockIdx.y * kQO;
  const long long nq = static_cast<long long>(a.B) * (a.T > 0 ? a.T : 1) * a.Hq;   // query rows
  const int tid = threadIdx.x, kg = tid >> 7, oq = 4 * (tid & 15), h0 = 4 * ((tid & 127) >> 4);
  pdl_trigger();                       // the partials kernel may launch now (it waits for this grid's results)
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid < 2 && a.sched) a.sched[tid] = 0;   // partials work counters
#pragma unroll
  for (int it = 0; it < kD * kQO / 4 / kQThreads; ++it) {
    const int v = tid + it * kQThreads, k = v / (kQO / 4), c = 4 * (v % (kQO / 4));
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c0 + c < nout) x = *reinterpret_cast<const float4*>(a.tab.wt + static_cast<long long>(k) * nout + c0 + c);
    *reinterpret_cast<float4*>(&ws[k][c]) = x;
  }
  {
    // row tid / 16, channels 8 (tid % 16) .. + 7: every load issued before the first store
    const int qr = tid >> 4, qc = 8 * (tid & 15);
    const bool in = r0 + qr < nq;
    float qv[8];
    if ((reinterpret_cast<uintptr_t>(a.q) & 15) == 0 && !a.f32) {
      const uint4 x = in ? *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + (r0 + qr) * kD + qc)
                         : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qv[2 * e] = __uint_as_float(xs[e] << 16);
        qv[2 * e + 1] = __uint_as_float(xs[e] & 0xFFFF0000u);
      }
    } else if ((reinterpret_cast<uintptr_t>(a.q) & 15) == 0) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + (r0 + qr) * kD + qc);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float4 x = in ? src[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[4 * j] = x.x;
        qv[4 * j + 1] = x.y;
        qv[4 * j + 2] = x.z;
        qv[4 * j + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) qv[j] = in ? load_q(a.q, a.f32, (r0 + qr) * kD + qc + j) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; j += 4)
      *reinterpret_cast<float4*>(&qs[qr][qc + j]) = make_float4(qv[j], qv[j + 1], qv[j + 2], qv[j + 3]);
  }
  __syncthreads();
  {
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.0f;
#pragma unroll 4
    for (int k = kg * kQK; k < kg * kQK + kQK; ++k) {
      const float4 w = *reinterpret_cast<const float4*>(&ws[k][oq]);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float qv = qs[h0 + r][k];
        acc[r][0] = fmaf(w.x, qv, acc[r][0]);
        acc[r][1] = fmaf(w.y, qv, acc[r][1]);
        acc[r][2] = fmaf(w.z, qv, acc[r][2]);
        acc[r][3] = fmaf(w.w, qv, acc[r][3]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
      *reinterpret_cast<float4*>(&ps[kg][h0 + r][oq]) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
  __syncthreads();
  // thread tid: head tid / 16, outputs 4 (tid % 16) .. + 3, the quarters summed in order
  const int hr = tid >> 4, oc = 4 * (tid & 15);
  float acc[4];
  {
    float4 x = *reinterpret_cast<const float4*>(&ps[0][hr][oc]);
#pragma unroll
    for (int g = 1; g < kQThreads / 128; ++g) {
      const float4 y = *reinterpret_cast<const float4*>(&ps[g][hr][oc]);
      x.x += y.x;
      x.y += y.y;
      x.z += y.z;
      x.w += y.w;
    }
    acc[0] = x.x, acc[1] = x.y, acc[2] = x.z, acc[3] = x.w;
  }
  if (c0 + oc < nout && r0 + hr < nq)
    *reinterpret_cast<float4*>(a.qprep + (r0 + hr) * nout + c0 + oc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  // fused step: this grid ends only after the append kernel before it (the
  // partials kernel, which waits for this grid, then sees the new token)
  if (a.chained) pdl_wait();
  if (!a.qfrag || a.m != kD) return;
  // fp16 fragments of the persistent partials kernel: this block's 64 outputs
  // hold, per head, 32 of its 128 words (slice 0/1: key pairs of channel group
  // 0/1 for every lane t; slice 2/3: u pairs of lanes t = 0,1 / 2,3)
  __shared__ __half hs[kQP][kQO];
  __shared__ __half hl[kQP][kQO];          // fp16 of the rounding remainder (q~ low parts)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __half h = __float2half_rn(acc[c]);
    hs[hr][oc + c] = h;
    hl[hr][oc + c] = __float2half_rn(acc[c] - __half2float(h));
  }
  __syncthreads();
  const int y = blockIdx.y;
  for (int idx = tid; idx < kQP * 32; idx += kQThreads) {
    const int h = idx >> 5, k = idx & 31;
    if (r0 + h >= nq) continue;
    int word, lo, hi;                        // word index in the head's 128, local offsets of its halves
    if (y < 2) {
      const int t = k >> 3, kk = 4 * y + ((k >> 1) & 3), e = k & 1;
      word = 32 * t + 2 * kk + e;
      lo = 16 * t + k_pair_channel(a.kl.g[y].bits, 2 * (kk & 3) + e);
      hi = lo + 1;
    } else {
      // u pair p = 2 st + h: projections 16h + st and 16h + 8 + st of word t,
      // the sign bits the kernel's prmt places in the pair at step st
      const int t = 2 * (y - 2) + (k >> 4), p = k & 15;
      word = 32 * t + 16 + p;
      lo = 32 * t + 16 * (p & 1) + (p >> 1) - 64 * (y - 2);
      hi = lo + 8;
    }
    a.qfrag[(r0 + h) * kQFragWords + word] = static_cast<uint32_t>(__half_as_ushort(hs[h][lo])) |
                                             (static_cast<uint32_t>(__half_as_ushort(hs[h][hi])) << 16);
    // q~ low parts of the key pairs: word 128 + 16 t + (2 kk + e), the same order
    if (y < 2) {
      const int t = k >> 3;
      a.qfrag[(r0 + h) * kQFragWords + 128 + 16 * t + (word - 32 * t)] =
          static_cast<uint32_t>(__half_as_ushort(hl[h][lo])) | (static_cast<uint32_t>(__half_as_ushort(hl[h][hi])) << 16);
    }
  }
}

// [q~; u] = W q for the tensor-core causal kernel, by query block: a CTA
// takes 64 rows r of one block (block rows r = t G + g of one sequence and KV
// head) x 128 outputs (q~, or u), with the whole K = 128 staged in shared
// memory; a thread holds 8 rows x 4 outputs, so three 16-byte shared loads feed
// 32 FMAs, each output summed over k in order as in qprep_kernel.  The outputs
// leave as fp16 words in tensor-memory column order (q~ hi pairs 0..63, q~ lo
// pairs 64..127, u pairs 128..191), word w of block row r at uint4
// (blk 48 + w / 4) 128 + r: restaged in shared memory so that the stores, like
// the causal kernel's loads (lane = block row), are 512 contiguous bytes.
constexpr int kQRRows = 64, kQROut = 128, kQRThreads = 256, kQRPad = kD + 4;
constexpr int kQRSmem = (kQRRows * kQRPad + kD * kQROut) * 4;

__global__ void __launch_bounds__(kQRThreads) qprep_rows_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float qsm[];
  float(*qs)[kQRPad] = reinterpret_cast<float(*)[kQRPad]>(qsm);
  float(*ws)[kQROut] = reinterpret_cast<float(*)[kQROut]>(qsm + kQRRows * kQRPad);
  const int nout = kD + a.m;
  const long long blk = blockIdx.x >> 1;
  const int xh = blockIdx.x & 1, c0 = blockIdx.y * kQROut;
  const int qb = static_cast<int>(blk % a.nqb);
  const long long bh = blk / a.nqb;
  const int h = static_cast<int>(bh % a.H);
  const long long b = bh / a.H;
  const int rows_all = a.T * a.G, rb = 128 * qb + 64 * xh;   // the CTA's first block row (as t G + g)
  const int tid = threadIdx.x;
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid < 2 && a.sched) a.sched[tid] = 0;   // partials work counters
  // every load of the W^T slice and the q rows issued before the first store
  {
    float4 wv[kD * kQROut / 4 / kQRThreads];
#pragma unroll
    for (int it = 0; it < kD * kQROut / 4 / kQRThreads; ++it) {
      const int v = tid + it * kQRThreads, k = v / (kQROut / 4), c = 4 * (v % (kQROut / 4));
      wv[it] = c0 + c < nout ? *reinterpret_cast<const float4*>(a.tab.wt + static_cast<long long>(k) * nout + c0 + c)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float qv[32];                                      // row tid / 4, channels 32 (tid % 4) ..
    const int qr = tid >> 2, qc = 32 * (tid & 3), rr = rb + qr;
    const bool in = rr < rows_all;
    const long long R = in ? (b * a.T + rr / a.G) * a.Hq + h * a.G + rr % a.G : 0;
    const bool vec = (reinterpret_cast<uintptr_t>(a.q) & 15) == 0;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
      if (!vec) {
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[j + e] = in ? load_q(a.q, a.f32, R * kD + qc + j + e) : 0.0f;
      } else if (a.f32) {
        const float* src = static_cast<const float*>(a.q) + R * kD + qc + j;
        const float4 x0 = in ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 x1 = in ? *reinterpret_cast<const float4*>(src + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[j] = x0.x; qv[j + 1] = x0.y; qv[j + 2] = x0.z; qv[j + 3] = x0.w;
        qv[j + 4] = x1.x; qv[j + 5] = x1.y; qv[j + 6] = x1.z; qv[j + 7] = x1.w;
      } else {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (in) x = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + R * kD + qc + j);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qv[j + 2 * e] = __uint_as_float(xs[e] << 16);
          qv[j + 2 * e + 1] = __uint_as_float(xs[e] & 0xFFFF0000u);
        }
      }
    }
#pragma unroll
    for (int it = 0; it < kD * kQROut / 4 / kQRThreads; ++it) {
      const int v = tid + it * kQRThreads, k = v / (kQROut / 4), c = 4 * (v % (kQROut / 4));
      *reinterpret_cast<float4*>(&ws[k][c]) = wv[it];
    }
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4*>(&qs[qr][qc + j]) = make_float4(qv[j], qv[j + 1], qv[j + 2], qv[j + 3]);
  }
  __syncthreads();
  const int tr = tid >> 5, to = tid & 31;          // rows 8 tr .. 8 tr + 7, outputs 4 to .. 4 to + 3
  float acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = 0.0f;
#pragma unroll 1
  for (int k0 = 0; k0 < kD; k0 += 4) {
    float4 w[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) w[kk] = *reinterpret_cast<const float4*>(&ws[k0 + kk][4 * to]);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float4 q4 = *reinterpret_cast<const float4*>(&qs[8 * tr + r][k0]);
      const float qk[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        acc[r][0] = fmaf(w[kk].x, qk[kk], acc[r][0]);
        acc[r][1] = fmaf(w[kk].y, qk[kk], acc[r][1]);
        acc[r][2] = fmaf(w[kk].z, qk[kk], acc[r][2]);
        acc[r][3] = fmaf(w[kk].w, qk[kk], acc[r][3]);
      }
    }
  }
  __syncthreads();                                 // the W^T slice is read: its space restages the words
  // staging: [group g (q~: hi 0..15, lo 16..31; u: 0..15)][row 64] x 16 bytes
  uint2* stg = reinterpret_cast<uint2*>(ws);
  const bool qt = c0 < kD;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int rl = 8 * tr + r;
    const __half2 h0 = __floats2half2_rn(acc[r][0], acc[r][1]), h1 = __floats2half2_rn(acc[r][2], acc[r][3]);
    stg[((to >> 1) * 64 + rl) * 2 + (to & 1)] =
        make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    if (qt) {
      const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
      const __half2 l0 = __floats2half2_rn(acc[r][0] - f0.x, acc[r][1] - f0.y);
      const __half2 l1 = __floats2half2_rn(acc[r][2] - f1.x, acc[r][3] - f1.y);
      stg[((16 + (to >> 1)) * 64 + rl) * 2 + (to & 1)] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
    }
  }
  __syncthreads();
  const int ng = qt ? 32 : 16, g0 = qt ? 0 : 32;   // groups of 4 words: this CTA's, and its first in the row
  uint4* dst = reinterpret_cast<uint4*>(a.qprep) + blk * 48 * 128 + 64 * xh;
  const uint4* src = reinterpret_cast<const uint4*>(ws);
  for (int i = tid; i < ng * 64; i += kQRThreads) dst[(g0 + i / 64) * 128 + i % 64] = src[i];
}

// Code of channel j from a vector's code words (the stored format of tq.h).
__device__ __forceinline__ int code_at(const unsigned* rec, int bh, int bl, int split, int j) {
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

template <int G>
__global__ void __launch_bounds__(kThreads) chunk_kernel(DecodeArgs a) {
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float qt_s[G][kD];
  __shared__ float u_s[G][kMaxM];
  __shared__ float ck_s[2][16];
  __shared__ float cv_s[2][16];
  __shared__ unsigned rec_s[4][32 * kRecStride];
  __shared__ float red_m[4][G];
  __shared__ float red_l[4][G];
  __shared__ float red_acc[4][G][kD];

  for (int idx = threadIdx.x; idx < G * kD; idx += kThreads) {
    int g = idx / kD, j = idx % kD;
    qt_s[g][j] = a.qprep[(static_cast<long long>(b) * a.Hq + h * G + g) * (kD + a.m) + j];
  }
  for (int idx = threadIdx.x; idx < G * a.m; idx += kThreads) {
    int g = idx / a.m, p = idx % a.m;
    u_s[g][p] = a.qprep[(static_cast<long long>(b) * a.Hq + h * G + g) * (kD + a.m) + kD + p];
  }
  if (threadIdx.x < 32) {
    int gi = threadIdx.x >> 4, k = threadIdx.x & 15;
    ck_s[gi][k] = a.kl.g[gi].c[k];
    cv_s[gi][k] = a.vl.g[gi].c[k];
  }
  int L = a.seq_lens[b] + a.len_add;
  if (L < 0 || L > a.max_seq_len || L > a.maxp * kPage) {
    if (threadIdx.x == 0 && chunk == 0 && h == 0) atomicOr(a.tab.err, kErrSeqLen);
    L = L < 0 ? 0 : L;
    L = L > a.max_seq_len ? a.max_seq_len : L;
    L = L > a.maxp * kPage ? a.maxp * kPage : L;
  }
  __syncthreads();

  const int t0 = chunk * a.chunk;
  const int t1 = min(t0 + a.chunk, L);
  const int kbh = a.kl.g[0].bits, kbl = a.kl.g[1].bits, ksplit = a.kl.split;
  const int vbh = a.vl.g[0].bits, vbl = a.vl.g[1].bits, vsplit = a.vl.split;
  const int kcw = a.kl.code_bytes / 4;
  const int swords = a.kl.qjl ? a.m / 32 : 0;
  const float qjl_scale = kSqrtHalfPi / static_cast<float>(a.m);
  unsigned* rec = rec_s[warp] + lane * kRecStride;

  float m_run[G], l_run[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[g][q] = 0.0f;
  }
  // this lane's 4 value channels
  const int vj0 = 4 * lane;
  const int vgrp = vj0 < vsplit ? 1 : 0;   // 1 -> hi group
  const float* cvt = cv_s[vgrp ? 0 : 1];

  for (int base = t0 + warp * 32; base < t1; base += 4 * 32) {
    const int t = base + lane;
    bool valid = t < t1;
    int page = 0;
    if (valid) {
      page = a.block_table[static_cast<long long>(b) * a.maxp + (t >> 4)];
      if (page < 0 || page >= a.num_pages) {
        atomicOr(a.tab.err, kErrPage);
        valid = false;
      }
    }
    const int slot = t & 15;
    float logit[G];
    if (valid) {
      const unsigned char* kb = a.kc + static_cast<long long>(page) * a.k_page_bytes +
                                static_cast<long long>(h) * a.kl.block_bytes;
      const unsigned* cw = reinterpret_cast<const unsigned*>(kb + slot * a.kl.code_bytes);
      for (int w = 0; w < kcw; ++w) rec[w] = cw[w];
      rec[kcw] = 0;
      float s1[G], s2[G];
#pragma unroll
      for (int g = 0; g < G; ++g) s1[g] = s2[g] = 0.0f;
      for (int j = 0; j < kD; ++j) {
        const int code = code_at(rec, kbh, kbl, ksplit, j);
        const float c = ck_s[j < ksplit ? 0 : 1][code];
#pragma unroll
        for (int g = 0; g < G; ++g) s1[g] = fmaf(c, qt_s[g][j], s1[g]);
      }
      const unsigned* sw = reinterpret_cast<const unsigned*>(kb + a.kl.off_signs + slot * (a.m / 8));
      for (int w = 0; w < swords; ++w) {
        const unsigned bitsw = sw[w];
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
          const bool pos = (bitsw >> i) & 1u;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float u = u_s[g][32 * w + i];
            s2[g] += pos ? u : -u;
          }
        }
      }
      const float nk = __half2float(reinterpret_cast<const __half*>(kb + a.kl.off_norm)[slot]);
      const float rk = a.kl.qjl ? __half2float(reinterpret_cast<const __half*>(kb + a.kl.off_rnorm)[slot]) : 0.0f;
#pragma unroll
      for (int g = 0; g < G; ++g)
        logit[g] = (nk * kInvSqrtD * s1[g] + qjl_scale * rk * s2[g]) * a.scale_log2;
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) logit[g] = -INFINITY;
    }
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mx = warp_max(logit[g]);
      const float m_new = fmaxf(m_run[g], mx);
      const float alpha = m_run[g] == -INFINITY ? 0.0f : exp2f(m_run[g] - m_new);
      p[g] = valid ? exp2f(logit[g] - m_new) : 0.0f;
      l_run[g] = l_run[g] * alpha + warp_sum(p[g]);
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[g][q] *= alpha;
      m_run[g] = m_new;
    }
    // value accumulation: every lane owns 4 channels, tokens go one by one
    const int ntok = min(32, t1 - base);
    for (int tt = 0; tt < ntok; ++tt) {
      const int ok = __shfl_sync(0xffffffffu, valid ? 1 : 0, tt);
      const int pg = __shfl_sync(0xffffffffu, page, tt);
      float w[G];
#pragma unroll
      for (int g = 0; g < G; ++g) w[g] = __shfl_sync(0xffffffffu, p[g], tt);
      if (!ok) continue;
      const int ts = (base + tt) & 15;
      const unsigned char* vb = a.vc + static_cast<long long>(pg) * a.v_page_bytes +
                                static_cast<long long>(h) * a.vl.block_bytes;
      const unsigned* vw = reinterpret_cast<const unsigned*>(vb + ts * a.vl.code_bytes);
      const float nv = __half2float(reinterpret_cast<const __half*>(vb + a.vl.off_norm)[ts]) * kInvSqrtD;
      float cv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) cv[q] = cvt[code_at(vw, vbh, vbl, vsplit, vj0 + q)];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float wg = w[g] * nv;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[g][q] = fmaf(wg, cv[q], acc[g][q]);
      }
    }
  }

#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp][g] = m_run[g];
      red_l[warp][g] = l_run[g];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) red_acc[warp][g][4 * lane + q] = acc[g][q];
  }
  __syncthreads();
  const int j = threadIdx.x;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][g]);
    float lsum = 0.0f, A = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (red_m[w][g] == -INFINITY) continue;
      const float sc = exp2f(red_m[w][g] - M);
      lsum = fmaf(sc, red_l[w][g], lsum);
      A = fmaf(sc, red_acc[w][g][j], A);
    }
    float* dst = a.part + ((static_cast<long long>(b) * a.Hq + h * G + g) * a.nchunks + chunk) * (kD + 2);
    if (j == 0) {
      dst[0] = M;
      dst[1] = lsum;
    }
    dst[2 + j] = A;
  }
}

// Decode merge (one query per row): log-sum-exp of the chunk partials, then
// o = Pi^T (acc / l).
// A block of eight warps takes 8 / WR rows, WR warps per row; warp k of a row
// reads chunks k, k + WR, ... (a lane holds four channels), every load of a
// batch of eight issued before the first use.  Each warp forms its row's
// maximum and weight sum itself (lane c holds chunks c, c + 32, ...), so only
// the channel sums cross warps.  What does not depend on the partials kernel
// is read before the grid dependency wait: Pi (staged in shared memory) and
// the rows' lengths.  The row's WR warps then rotate it back, warp k taking
// rows 128 k / WR .. of Pi.
constexpr int kMDWarps = 8;
constexpr int kMDBatch = 8;                           // chunks in flight per warp
constexpr int kMDSmem = (kD * kD + 2 * kMDWarps * kD) * 4;   // Pi, the warps' channel sums, their rotated parts

template <int WR>
__global__ void __launch_bounds__(32 * kMDWarps) merge_dec_kernel(DecodeArgs a, long long rows) {
  extern __shared__ __align__(16) float mds[];
  float(*pis)[kD] = reinterpret_cast<float(*)[kD]>(mds);
  float(*cs)[kD] = reinterpret_cast<float(*)[kD]>(mds + kD * kD);                  // channel sums, per warp
  float(*rs)[kD] = reinterpret_cast<float(*)[kD]>(mds + kD * kD + kMDWarps * kD);  // rotated parts, per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = warp % WR, w0 = warp - k;              // this warp's share of its row, the row's first warp
  const long long row = static_cast<long long>(blockIdx.x) * (kMDWarps / WR) + warp / WR;
  const bool live = row < rows;
#pragma unroll
  for (int v4 = 0; v4 < kD * kD / 4 / (32 * kMDWarps); ++v4) {
    const int v = tid + v4 * 32 * kMDWarps;
    *reinterpret_cast<float4*>(&pis[0][0] + 4 * v) = __ldg(reinterpret_cast<const float4*>(a.tab.pi) + v);
  }
  int nc = 0;
  if (live) {
    int L = a.seq_lens[row / a.Hq] + a.len_add;
    L = L < 0 ? 0 : L;
    L = L > a.max_seq_len ? a.max_seq_len : L;
    L = L > a.maxp * kPage ? a.maxp * kPage : L;
    nc = min(a.nchunks, (L + a.chunk - 1) / a.chunk);
  }
  pdl_wait();                          // the partials kernel before it has completed
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, l = 0.0f;
  if (live) {
    const float* P = a.part + row * a.nchunks * (kD + 2);
    // this warp's first batch of chunks and the row's (max, sum) pairs, all issued before any use
    float2 x[kMDBatch][2];
    float mx[kMDBatch];
#pragma unroll
    for (int j = 0; j < kMDBatch; ++j) {
      const int c = k + WR * j;
      x[j][0] = x[j][1] = make_float2(0.f, 0.f);
      mx[j] = -INFINITY;
      if (c < nc) {
        const float* pc = P + static_cast<long long>(c) * (kD + 2);
        mx[j] = pc[0];
        x[j][0] = *reinterpret_cast<const float2*>(pc + 2 + 4 * lane);
        x[j][1] = *reinterpret_cast<const float2*>(pc + 4 + 4 * lane);
      }
    }
    float2 ml = make_float2(-INFINITY, 0.0f);
    if (lane < nc) ml = *reinterpret_cast<const float2*>(P + static_cast<long long>(lane) * (kD + 2));
    float M = ml.x;
    for (int c = lane + 32; c < nc; c += 32) M = fmaxf(M, P[static_cast<long long>(c) * (kD + 2)]);
    M = warp_max(M);
    if (M > -INFINITY) {
      l = lane < nc ? exp2f(ml.x - M) * ml.y : 0.0f;
      for (int c = lane + 32; c < nc; c += 32) {
        const float2 m2 = *reinterpret_cast<const float2*>(P + static_cast<long long>(c) * (kD + 2));
        l = fmaf(exp2f(m2.x - M), m2.y, l);
      }
      for (int cb = 0;; cb += kMDBatch) {
#pragma unroll
        for (int j = 0; j < kMDBatch; ++j) {
          const float w = exp2f(mx[j] - M);          // 0 past the row's chunks (-inf)
          acc[0] = fmaf(w, x[j][0].x, acc[0]);
          acc[1] = fmaf(w, x[j][0].y, acc[1]);
          acc[2] = fmaf(w, x[j][1].x, acc[2]);
          acc[3] = fmaf(w, x[j][1].y, acc[3]);
        }
        if (k + WR * (cb + kMDBatch) >= nc) break;
#pragma unroll
        for (int j = 0; j < kMDBatch; ++j) {       // the next batch
          const int c = k + WR * (cb + kMDBatch + j);
          x[j][0] = x[j][1] = make_float2(0.f, 0.f);
          mx[j] = -INFINITY;
          if (c < nc) {
            const float* pc = P + static_cast<long long>(c) * (kD + 2);
            mx[j] = pc[0];
            x[j][0] = *reinterpret_cast<const float2*>(pc + 2 + 4 * lane);
            x[j][1] = *reinterpret_cast<const float2*>(pc + 4 + 4 * lane);
          }
        }
      }
      l = warp_sum(l);
    }
  }
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  *reinterpret_cast<float4*>(&cs[warp][4 * lane]) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  __syncthreads();                     // Pi staged, every warp's channel sums written
  // o = Pi^T o~ over rows i of Pi in [i0, i0 + 128 / WR): o~_i summed over the row's warps
  constexpr int NI = kD / WR;
  const int i0 = k * NI;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int i = i0; i < i0 + NI; ++i) {
    const float4 p = *reinterpret_cast<const float4*>(&pis[i][4 * lane]);
    float xo = cs[w0][i];
#pragma unroll
    for (int r = 1; r < WR; ++r) xo += cs[w0 + r][i];
    o[0] = fmaf(p.x, xo, o[0]);
    o[1] = fmaf(p.y, xo, o[1]);
    o[2] = fmaf(p.z, xo, o[2]);
    o[3] = fmaf(p.w, xo, o[3]);
  }
  if (WR > 1) {
    *reinterpret_cast<float4*>(&rs[warp][4 * lane]) = make_float4(o[0], o[1], o[2], o[3]);
    __syncthreads();
    if (k != 0) return;
#pragma unroll
    for (int r = 1; r < WR; ++r) {
      const float4 q = *reinterpret_cast<const float4*>(&rs[w0 + r][4 * lane]);
      o[0] += q.x;
      o[1] += q.y;
      o[2] += q.z;
      o[3] += q.w;
    }
  }
  if (live) *reinterpret_cast<float4*>(a.out + row * kD + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
}

// Merge for many query rows (causal attention: B T Hq rows): a block takes 32
// rows.  Each warp combines the chunk partials of four rows (log-sum-exp of
// the chunk maxima, then the weighted sums; a lane holds four channels) into
// o~ = acc / l in shared memory; then the block rotates its 32 rows back at
// once, o = Pi^T o~, reading Pi once per 32 rows instead of once per row.
constexpr int kMRRows = 32;
constexpr int kMRThreads = 256;

__global__ void __launch_bounds__(kMRThreads) merge_rows_kernel(DecodeArgs a, long long rows) {
  pdl_wait();                          // the partials kernel before it has completed
  __shared__ __align__(16) float os[kMRRows][kD + 4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long r0 = static_cast<long long>(blockIdx.x) * kMRRows;
  // a warp's four rows together, so that their loads are in flight at once;
  // lane c holds chunk c's weight (chunks c, c + 32, ... in turn)
  constexpr int R = kMRRows / (kMRThreads / 32);
  const float* P[R];
  int nc[R];
  float M[R], l[R], acc[R][4];
  int ncmax = 0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const long long row = r0 + warp * R + i;
    nc[i] = 0;
    P[i] = a.part;
    if (row < rows) {
      // row (b, t, h) attends positions [0, seq_lens[b] + t]
      int L = a.seq_lens[row / a.Hq / a.T] + static_cast<int>((row / a.Hq) % a.T) + 1;
      L = L < 0 ? 0 : L;
      L = L > a.max_seq_len ? a.max_seq_len : L;
      L = L > a.maxp * kPage ? a.maxp * kPage : L;
      nc[i] = min(a.nchunks, (L + a.chunk - 1) / a.chunk);
      P[i] = a.part + row * a.nchunks * (kD + 2);
    }
    ncmax = max(ncmax, nc[i]);
    M[i] = -INFINITY;
    l[i] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.0f;
  }
  for (int cb = 0; cb < ncmax; cb += 32) {
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (cb + lane < nc[i]) M[i] = fmaxf(M[i], P[i][static_cast<long long>(cb + lane) * (kD + 2)]);
  }
#pragma unroll
  for (int i = 0; i < R; ++i) M[i] = warp_max(M[i]);
  for (int cb = 0; cb < ncmax; cb += 32) {
    float w[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      w[i] = 0.0f;
      if (cb + lane < nc[i]) {
        const float2 ml = *reinterpret_cast<const float2*>(P[i] + static_cast<long long>(cb + lane) * (kD + 2));
        w[i] = exp2f(ml.x - M[i]);
        l[i] = fmaf(w[i], ml.y, l[i]);
      }
    }
    const int n = min(32, ncmax - cb);
    for (int j0 = 0; j0 < n; j0 += 2) {
      float2 x[R][2][2];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int c = cb + j0 + jj;
          x[i][jj][0] = x[i][jj][1] = make_float2(0.f, 0.f);
          if (j0 + jj < n && c < nc[i]) {
            const float* pc = P[i] + static_cast<long long>(c) * (kD + 2) + 2 + 4 * lane;
            x[i][jj][0] = *reinterpret_cast<const float2*>(pc);
            x[i][jj][1] = *reinterpret_cast<const float2*>(pc + 2);
          }
        }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float wj = __shfl_sync(0xffffffffu, w[i], (j0 + jj) & 31);
          acc[i][0] = fmaf(wj, x[i][jj][0].x, acc[i][0]);
          acc[i][1] = fmaf(wj, x[i][jj][0].y, acc[i][1]);
          acc[i][2] = fmaf(wj, x[i][jj][1].x, acc[i][2]);
          acc[i][3] = fmaf(wj, x[i][jj][1].y, acc[i][3]);
        }
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const float lt = warp_sum(l[i]);
    const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
    *reinterpret_cast<float4*>(&os[warp * R + i][4 * lane]) =
        make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
  }
  __syncthreads();
  // thread: rows 4 rg .. 4 rg + 3, output channels 4 cg .. 4 cg + 3
  const int rg = tid >> 5, cg = tid & 31;
  float o[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[r][c] = 0.0f;
#pragma unroll 4
  for (int i = 0; i < kD; ++i) {
    const float4 p = __ldg(reinterpret_cast<const float4*>(a.tab.pi + i * kD + 4 * cg));
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float x = os[4 * rg + r][i];
      o[r][0] = fmaf(p.x, x, o[r][0]);
      o[r][1] = fmaf(p.y, x, o[r][1]);
      o[r][2] = fmaf(p.z, x, o[r][2]);
      o[r][3] = fmaf(p.w, x, o[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const long long row = r0 + 4 * rg + r;
    if (row < rows)
      *reinterpret_cast<float4*>(a.out + row * kD + 4 * cg) = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
  }
}

// Merge for the tensor-core causal kernel, whose partials are stored by query
// block: (max, sum, acc[128]) of block row r for chunk c at float
// ((blk nchunks + c) 130 + f) 128 + r.  A block takes 32 rows of a query
// block: lane = row, warp w the channels 16 w .. 16 w + 15, so that every load
// of a warp is 128 contiguous bytes; then o = Pi^T o~ for the 32 rows.
constexpr int kMBThreads = 512;

__global__ void __launch_bounds__(kMBThreads) merge_blk_kernel(DecodeArgs a) {
  pdl_wait();                          // the partials kernel before it has completed
  __shared__ __align__(16) float os[32][kD + 4];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long blk = blockIdx.x >> 2;
  const int sub = blockIdx.x & 3;
  const int qb = static_cast<int>(blk % a.nqb);
  const long long bh = blk / a.nqb;
  const int h = static_cast<int>(bh % a.H);
  const long long b = bh / a.H;
  const int rows_all = a.T * a.G;
  {
    const int rr = 128 * qb + 32 * sub + lane;
    int nc = 0;
    if (rr < rows_all) {
      int L = a.seq_lens[b] + rr / a.G + 1;          // row t G + g attends positions [0, start + t]
      L = L < 0 ? 0 : L;
      L = L > a.max_seq_len ? a.max_seq_len : L;
      L = L > a.maxp * kPage ? a.maxp * kPage : L;
      nc = min(a.nchunks, (L + a.chunk - 1) / a.chunk);
    }
    const float* pb = a.part + blk * a.nchunks * (kD + 2) * 128 + 32 * sub + lane;
    constexpr long long kCS = (kD + 2) * 128;          // floats between a row's chunks
    int ncw = nc;                                      // the warp's largest chunk count
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ncw = max(ncw, __shfl_xor_sync(0xffffffffu, ncw, o));
    // loads in batches of eight chunks (maxima) and four chunks (sums and this warp's channels)
    float M = -INFINITY;
    for (int c0 = 0; c0 < ncw; c0 += 8) {
      float mv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mv[j] = c0 + j < nc ? pb[(c0 + j) * kCS] : -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) M = fmaxf(M, mv[j]);
    }
    float l = 0.0f, acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    for (int c0 = 0; c0 < ncw; c0 += 4) {
      float mv[4], lv[4], xv[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool in = c0 + j < nc;
        const float* pc = pb + (c0 + j) * kCS;
        mv[j] = in ? pc[0] : -INFINITY;
        lv[j] = in ? pc[128] : 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) xv[j][k] = in ? pc[(2 + 8 * warp + k) * 128] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = c0 + j < nc ? exp2f(mv[j] - M) : 0.0f;
        l = fmaf(w, lv[j], l);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = fmaf(w, xv[j][k], acc[k]);
      }
    }
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    *reinterpret_cast<float4*>(&os[lane][8 * warp]) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<float4*>(&os[lane][8 * warp + 4]) = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
  __syncthreads();
  const int rg = tid >> 5, cg = tid & 31;            // rows 2 rg, 2 rg + 1, output channels 4 cg .. 4 cg + 3
  float o[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[r][c] = 0.0f;
#pragma unroll 4
  for (int i = 0; i < kD; ++i) {
    const float4 p = __ldg(reinterpret_cast<const float4*>(a.tab.pi + i * kD + 4 * cg));
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float x = os[2 * rg + r][i];
      o[r][0] = fmaf(p.x, x, o[r][0]);
      o[r][1] = fmaf(p.y, x, o[r][1]);
      o[r][2] = fmaf(p.z, x, o[r][2]);
      o[r][3] = fmaf(p.w, x, o[r][3]);
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int rr = 128 * qb + 32 * sub + 2 * rg + r;
    if (rr >= rows_all) continue;
    const long long row = (b * a.T + rr / a.G) * a.Hq + h * a.G + rr % a.G;
    *reinterpret_cast<float4*>(a.out + row * kD + 4 * cg) = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
  }
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.nchunks, a.H, a.B);
  chunk_kernel<G><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int stages, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if ((stages & TQ_STAGE_QPREP) && a.qhalf) {
    const long long nblk = static_cast<long long>(a.B) * a.H * a.nqb;
    const dim3 grid(static_cast<unsigned>(2 * nblk), static_cast<unsigned>((kD + a.m + kQROut - 1) / kQROut));
    static std::atomic<unsigned long long> configured{0};   // q rows and the W^T slice take 99 KB
    e = smem_attr_once(qprep_rows_kernel, kQRSmem, configured);
    if (e != cudaSuccess) return e;
    qprep_rows_kernel<<<grid, kQRThreads, kQRSmem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (stages & TQ_STAGE_QPREP) {
    const dim3 grid(static_cast<unsigned>((static_cast<long long>(a.B) * (a.T > 0 ? a.T : 1) * a.Hq + kQP - 1) / kQP),
                    static_cast<unsigned>((kD + a.m + kQO - 1) / kQO));
    static std::atomic<unsigned long long> configured{0};   // the W slice, q rows and partial tiles take 81 KB
    e = smem_attr_once(qprep_kernel, kQprepSmem, configured);
    if (e != cudaSuccess) return e;
    if (a.chained) {
      e = launch_pdl(qprep_kernel, grid, dim3(kQThreads), static_cast<size_t>(kQprepSmem), s, a);
    } else {
      qprep_kernel<<<grid, kQThreads, kQprepSmem, s>>>(a);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  if (stages & TQ_STAGE_PARTIALS) {
    cudaError_t em = cudaSuccess;
    if (launch_partials_lut(a, s, &em)) {
      if (em != cudaSuccess) return em;
    } else {
    switch (a.G) {
      case 1: e = launch_g<1>(a, s); break;
      case 2: e = launch_g<2>(a, s); break;
      case 3: e = launch_g<3>(a, s); break;
      case 4: e = launch_g<4>(a, s); break;
      case 5: e = launch_g<5>(a, s); break;
      case 6: e = launch_g<6>(a, s); break;
      case 7: e = launch_g<7>(a, s); break;
      case 8: e = launch_g<8>(a, s); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    }
  }
  if (stages & TQ_STAGE_MERGE) {
    if (a.T > 0 && a.qhalf) {
      const long long nblk = static_cast<long long>(a.B) * a.H * a.nqb;
      e = launch_pdl(merge_blk_kernel, dim3(static_cast<unsigned>(4 * nblk)), dim3(kMBThreads), 0, s, a);
    } else if (a.T > 0) {
      const long long rows = static_cast<long long>(a.B) * a.T * a.Hq;
      e = launch_pdl(merge_rows_kernel, dim3(static_cast<unsigned>((rows + kMRRows - 1) / kMRRows)), dim3(kMRThreads),
                     0, s, a, rows);
    } else {
      // warps per row: a batch of eight chunks per warp for up to 32 chunks, then
      // as many warps as keep the batches (and the rows per block) few
      const long long rows = static_cast<long long>(a.B) * a.Hq;
      const int wr = a.nchunks <= 8 ? 1 : a.nchunks <= 16 ? 2 : a.nchunks <= 32 ? 4 : 8;
      const dim3 grid(static_cast<unsigned>((rows + kMDWarps / wr - 1) / (kMDWarps / wr)));
      static std::atomic<unsigned long long> configured[4];   // Pi and the warps' sums take 72 KB
      switch (wr) {
        case 1: e = smem_attr_once(merge_dec_kernel<1>, kMDSmem, configured[0]); break;
        case 2: e = smem_attr_once(merge_dec_kernel<2>, kMDSmem, configured[1]); break;
        case 4: e = smem_attr_once(merge_dec_kernel<4>, kMDSmem, configured[2]); break;
        default: e = smem_attr_once(merge_dec_kernel<8>, kMDSmem, configured[3]); break;
      }
      if (e != cudaSuccess) return e;
      const size_t sm = static_cast<size_t>(kMDSmem);
      switch (wr) {
        case 1: e = launch_pdl(merge_dec_kernel<1>, grid, dim3(32 * kMDWarps), sm, s, a, rows); break;
        case 2: e = launch_pdl(merge_dec_kernel<2>, grid, dim3(32 * kMDWarps), sm, s, a, rows); break;
        case 4: e = launch_pdl(merge_dec_kernel<4>, grid, dim3(32 * kMDWarps), sm, s, a, rows); break;
        default: e = launch_pdl(merge_dec_kernel<8>, grid, dim3(32 * kMDWarps), sm, s, a, rows); break;
      }
    }
  }
  return e;
}

}  // namespace tq
