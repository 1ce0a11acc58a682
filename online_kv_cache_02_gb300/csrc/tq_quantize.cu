// Online quantize-and-append kernel.
//
// [P2] "생각정리 209 (TurboQuant)", stage 1 and stage 2; [P4] riverfrot.github.io
// "TurboQuant란 무엇이며…", §4.1 (x~ = R x/||x||), §4.2 (per-coordinate
// Lloyd-Max lookup), §4.3 (residual r = x - Q^-1(Q(x)), 1-bit sign sketch of a
// random projection of r), §3.1 (fixed-size blocks addressed by a block table).
//
// Per tile of 32 vectors (one CTA, persistent over tiles, Pi^T and S^T resident
// in shared memory):
//   1. x tile -> shared (transposed), ||x||^2 as an exact double-float sum
//   2. y = Pi x on the fp32 pipes (4x4 register tile per thread)
//   3. u = sqrt(d) y / ||x||, code = #{k : u >= t_k}; a u within 2e-5 of a
//      boundary is re-decided from y and ||x|| recomputed in fp64
//   4. keys: r = y - fp16(||x||)/sqrt(d) c[code]; z = S r (fp32); sign = z >= 0;
//      if any |z_i| < 5e-5 ||r|| the whole vector's r, z and ||r|| are redone
//      in fp64 (the fp32 residual carries the cancellation error of y - y^)
//   5. bit-pack codes / signs, fp16 norms, store at (page, slot, head).
// fp32 error of the fast path is ~1e-7 in u units and ~1e-6 ||r|| for z, so
// the guards sit 100x and 30x beyond it: the stored codes and signs are the
// ones exact arithmetic gives, except for values within ~1e-13 of a boundary.

#include "tq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace tq {
namespace {

constexpr int kTile = 32;
constexpr int kThreads = 256;
constexpr int kXS = 36;            // padded row stride (floats) of the transposed tiles
constexpr float kCodeGuard = 2e-5f;
constexpr float kSignGuard = 5e-5f;

// ---- double-float helpers (error-free transformations) ----------------------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  e = b - (s - a);
}
__device__ __forceinline__ void df_add(float& h, float& l, float bh, float bl) {
  float s, e;
  two_sum(h, bh, s, e);
  e += l + bl;
  fast_two_sum(s, e, h, l);
}

// fp16 round-to-nearest-even of the double-float value hi + lo (hi >= 0).
__device__ __half df_to_half(float hi, float lo) {
  __half h = __float2half_rn(hi);
  float back = __half2float(h);
  if (back == hi || lo == 0.0f || isinf(back)) return h;
  unsigned short bits = __half_as_ushort(h);
  __half nb = __ushort_as_half(hi > back ? static_cast<unsigned short>(bits + 1)
                                         : static_cast<unsigned short>(bits - 1));
  float nbf = __half2float(nb);
  float mid = 0.5f * (back + nbf);
  if (hi != mid) return h;                 // not on a tie: hi rounds like hi + lo
  bool up = lo > 0.0f;                     // tie broken by the low part
  bool nb_is_up = nbf > back;
  return (up == nb_is_up) ? nb : h;
}

__device__ __forceinline__ float load_x(const void* x, bool f32, long long idx) {
  if (f32) return static_cast<const float*>(x)[idx];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[idx]);
}

struct Smem {
  float* pit;     // [128][128]
  float* st;      // [128][128]  (S^T, columns >= m unused)
  float* xt;      // [128][kXS]
  float* rt;      // [128][kXS]
  unsigned char* codes;   // [32][128]
  unsigned char* snib;    // [32][32]
  double* r64;    // [8 warps][128]
  float* npart;   // [8][32][2]
  float* nhi;     // [32]
  float* nlo;
  float* scale;
  float* n16f;
  float* rho2;
  unsigned* sflag;   // [32]
  unsigned* sword;   // [32][4] refined sign words
  unsigned short* n16;   // [32]
  unsigned short* r16;   // [32]
};

template <bool KEY>
size_t smem_bytes() {
  size_t b = 0;
  b += 128 * 128 * 4;                 // pit
  if (KEY) b += 128 * 128 * 4;        // st
  b += 128 * kXS * 4;                 // xt
  if (KEY) b += 128 * kXS * 4;        // rt
  b += 32 * 128;                      // codes
  b += 32 * 32;                       // snib
  if (KEY) b += 8 * 128 * 8;          // r64
  b += 8 * 32 * 2 * 4;                // npart
  b += 5 * 32 * 4;                    // nhi, nlo, scale, n16f, rho2
  b += 32 * 4 + 32 * 4 * 4;           // sflag, sword
  b += 2 * 32 * 2;                    // n16, r16
  return b + 64;
}

template <bool KEY>
__device__ Smem carve(unsigned char* p) {
  Smem s;
  auto take = [&](size_t n) { unsigned char* r = p; p += (n + 15) & ~size_t(15); return r; };
  s.pit = reinterpret_cast<float*>(take(128 * 128 * 4));
  s.st = KEY ? reinterpret_cast<float*>(take(128 * 128 * 4)) : nullptr;
  s.xt = reinterpret_cast<float*>(take(128 * kXS * 4));
  s.rt = KEY ? reinterpret_cast<float*>(take(128 * kXS * 4)) : nullptr;
  s.r64 = KEY ? reinterpret_cast<double*>(take(8 * 128 * 8)) : nullptr;
  s.codes = take(32 * 128);
  s.snib = take(32 * 32);
  s.npart = reinterpret_cast<float*>(take(8 * 32 * 2 * 4));
  s.nhi = reinterpret_cast<float*>(take(32 * 4));
  s.nlo = reinterpret_cast<float*>(take(32 * 4));
  s.scale = reinterpret_cast<float*>(take(32 * 4));
  s.n16f = reinterpret_cast<float*>(take(32 * 4));
  s.rho2 = reinterpret_cast<float*>(take(32 * 4));
  s.sflag = reinterpret_cast<unsigned*>(take(32 * 4));
  s.sword = reinterpret_cast<unsigned*>(take(32 * 4 * 4));
  s.n16 = reinterpret_cast<unsigned short*>(take(32 * 2));
  s.r16 = reinterpret_cast<unsigned short*>(take(32 * 2));
  return s;
}

// Stored 24-bit octet of eight 3-bit codes: channels 0-5 in nibbles (bits
// 4i..4i+2), channel 6 in bits 3/11/19 and channel 7 in bits 7/15/23.
__device__ __forceinline__ unsigned octet3(const unsigned char* c) {
  unsigned v = 0;
  for (int i = 0; i < 6; ++i) v |= static_cast<unsigned>(c[i]) << (4 * i);
  for (int q = 0; q < 3; ++q) {
    v |= ((c[6] >> q) & 1u) << (8 * q + 3);
    v |= ((c[7] >> q) & 1u) << (8 * q + 7);
  }
  return v;
}

// Stored 4-bit value: sign-magnitude (bit 3 = negative half, bits 0-2 = rank of |centroid|).
__device__ __forceinline__ unsigned stored4(unsigned c) { return c >= 8 ? c - 8 : 15 - c; }

// 32-bit word w of a vector's code area, from one byte per channel.
__device__ unsigned pack_code_word(const KindLayout& L, const unsigned char* codes, int w) {
  const int lo = 32 * w, hi = lo + 32;
  unsigned word = 0;
  for (int grp = 0; grp < 2; ++grp) {
    const int b = L.g[grp].bits;
    const int c0 = grp ? L.split : 0;
    const int n = grp ? kD - L.split : L.split;
    const int base = grp ? L.split * L.g[0].bits : 0;
    if (n == 0 || base >= hi || base + n * b <= lo) continue;
    if (b == 3) {
      for (int o = 0; o < n / 8; ++o) {
        const int off = base + 24 * o;
        if (off >= hi || off + 24 <= lo) continue;
        const unsigned long long v = octet3(codes + c0 + 8 * o);
        const int sh = off - lo;
        word |= sh >= 0 ? static_cast<unsigned>(v << sh) : static_cast<unsigned>(v >> (-sh));
      }
    } else {
      const int cs = lo > base ? (lo - base) / b : 0;
      const int ce = min(n, (hi - base + b - 1) / b);
      for (int c = cs; c < ce; ++c) {
        unsigned long long v = codes[c0 + c];
        if (b == 4) v = stored4(static_cast<unsigned>(v));
        const int sh = base + b * c - lo;
        word |= sh >= 0 ? static_cast<unsigned>(v << sh) : static_cast<unsigned>(v >> (-sh));
      }
    }
  }
  return word;
}

template <bool KEY>
__global__ void __launch_bounds__(kThreads, 1) quantize_kernel(QuantizeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem sm = carve<KEY>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const KindLayout& L = a.lay;
  const float inv_sqrt_d = 0.08838834764831845f;     // 1/sqrt(128)
  const double inv_sqrt_d64 = 1.0 / sqrt(128.0);
  const double sqrt_d64 = sqrt(128.0);

  for (int i = tid; i < 128 * 128 / 4; i += kThreads)
    reinterpret_cast<float4*>(sm.pit)[i] = reinterpret_cast<const float4*>(a.tab.pit)[i];
  if (KEY) {
    for (int i = tid; i < 128 * 128; i += kThreads) {
      int j = i >> 7, c = i & 127;
      sm.st[i] = c < a.m ? a.tab.st[j * a.m + c] : 0.0f;
    }
  }
  __syncthreads();

  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  const long long ntiles = (nvec + kTile - 1) / kTile;
  for (long long tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const long long v0 = tile * kTile;
    // 1. x tile (transposed) and double-float partial norms
    {
      const int v = lane, kc = warp;
      const long long gv = v0 + v;
      float sh = 0.0f, sl = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        int k = kc * 16 + q;
        float xv = gv < nvec ? load_x(a.x, a.f32, gv * kD + k) : 0.0f;
        sm.xt[k * kXS + v] = xv;
        float p = xv * xv;
        float e = fmaf(xv, xv, -p);
        float s, t;
        two_sum(sh, p, s, t);
        sh = s;
        sl += t + e;
      }
      sm.npart[(kc * 32 + v) * 2 + 0] = sh;
      sm.npart[(kc * 32 + v) * 2 + 1] = sl;
      if (tid < 32) sm.sflag[tid] = 0;
    }
    __syncthreads();
    if (tid < 32) {
      float h = 0.0f, l = 0.0f;
      for (int kc = 0; kc < 8; ++kc) df_add(h, l, sm.npart[(kc * 32 + tid) * 2], sm.npart[(kc * 32 + tid) * 2 + 1]);
      float nh = 0.0f, nl = 0.0f;
      if (h > 0.0f) {
        float r = sqrtf(h);
        float res = fmaf(-r, r, h) + l;
        fast_two_sum(r, res / (2.0f * r), nh, nl);
      }
      sm.nhi[tid] = nh;
      sm.nlo[tid] = nl;
      sm.scale[tid] = nh > 0.0f ? 11.313708498984761f / nh : 0.0f;   // sqrt(128) / ||x||
      __half n16 = df_to_half(nh, nl);
      sm.n16[tid] = __half_as_ushort(n16);
      sm.n16f[tid] = __half2float(n16);
    }
    __syncthreads();

    // 2. y = Pi x: thread owns vectors 4*warp..+3, outputs 4*lane..+3
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
#pragma unroll 8
    for (int k = 0; k < 128; ++k) {
      float4 p = *reinterpret_cast<const float4*>(&sm.pit[k * 128 + 4 * lane]);
      float4 xx = *reinterpret_cast<const float4*>(&sm.xt[k * kXS + 4 * warp]);
      float xa[4] = {xx.x, xx.y, xx.z, xx.w};
      float pa[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int vi = 0; vi < 4; ++vi)
#pragma unroll
        for (int oi = 0; oi < 4; ++oi) acc[vi][oi] = fmaf(pa[oi], xa[vi], acc[vi][oi]);
    }

    // 3. codes (+ fp64 re-decision near boundaries); keys: residual
    float rpart[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int vi = 0; vi < 4; ++vi) {
      const int v = 4 * warp + vi;
      const bool valid = v0 + v < nvec;
      const float sc = sm.scale[v];
#pragma unroll
      for (int oi = 0; oi < 4; ++oi) {
        const int i = 4 * lane + oi;
        const GroupBook& gb = L.g[i < L.split ? 0 : 1];
        float u = acc[vi][oi] * sc;
        int code = 0;
        float mind = INFINITY;
        for (int k = 0; k < gb.nb; ++k) {
          code += u >= gb.t[k];
          mind = fminf(mind, fabsf(u - gb.t[k]));
        }
        if (valid && mind < kCodeGuard) {
          double y64 = 0.0;
          for (int k = 0; k < 128; ++k) y64 = fma(a.tab.pi64[i * 128 + k], static_cast<double>(sm.xt[k * kXS + v]), y64);
          double n64 = static_cast<double>(sm.nhi[v]) + static_cast<double>(sm.nlo[v]);
          double u64 = n64 > 0.0 ? sqrt_d64 * y64 / n64 : 0.0;
          code = 0;
          for (int k = 0; k < gb.nb; ++k) code += u64 >= gb.t64[k];
          atomicAdd(&a.tab.counters[0], 1ULL);
        }
        sm.codes[v * 128 + i] = static_cast<unsigned char>(code);
        if (KEY) {
          float r = fmaf(-sm.n16f[v] * inv_sqrt_d, gb.c[code], acc[vi][oi]);
          sm.rt[i * kXS + v] = r;
          rpart[vi] = fmaf(r, r, rpart[vi]);
        }
      }
    }
    if (KEY) {
#pragma unroll
      for (int vi = 0; vi < 4; ++vi) {
        float s = rpart[vi];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) sm.rho2[4 * warp + vi] = s;
      }
      __syncthreads();
      // 4. z = S r for projections 4*lane..+3
      float z[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) z[i][j] = 0.0f;
#pragma unroll 8
      for (int j = 0; j < 128; ++j) {
        float4 s4 = *reinterpret_cast<const float4*>(&sm.st[j * 128 + 4 * lane]);
        float4 rr = *reinterpret_cast<const float4*>(&sm.rt[j * kXS + 4 * warp]);
        float ra[4] = {rr.x, rr.y, rr.z, rr.w};
        float sa[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int vi = 0; vi < 4; ++vi)
#pragma unroll
          for (int oi = 0; oi < 4; ++oi) z[vi][oi] = fmaf(sa[oi], ra[vi], z[vi][oi]);
      }
#pragma unroll
      for (int vi = 0; vi < 4; ++vi) {
        const int v = 4 * warp + vi;
        const float guard = kSignGuard * sqrtf(sm.rho2[v]);
        unsigned nib = 0;
        bool near = false;
#pragma unroll
        for (int oi = 0; oi < 4; ++oi) {
          nib |= (z[vi][oi] >= 0.0f ? 1u : 0u) << oi;
          near |= (4 * lane + oi < a.m) && fabsf(z[vi][oi]) < guard;
        }
        sm.snib[v * 32 + lane] = static_cast<unsigned char>(nib);
        unsigned any = __ballot_sync(0xffffffffu, near);
        if (lane == 0 && any) sm.sflag[v] = 1u;
      }
    }
    __syncthreads();

    // 5. per-vector finalisation: warp handles vectors warp, warp+8, ...
    for (int r = 0; r < 4; ++r) {
      const int v = warp + 8 * r;
      const long long gv = v0 + v;
      if (gv >= nvec) continue;
      const int h = static_cast<int>(gv % a.H);
      const long long bt = gv / a.H;
      const int t = static_cast<int>(bt % a.n_new);
      const int b = static_cast<int>(bt / a.n_new);
      bool refine = KEY && L.qjl && sm.sflag[v];
      unsigned short r16 = 0;
      if (KEY && L.qjl) {
        if (refine) {
          // fp64 residual, projections and residual norm for this vector
          double* r64 = sm.r64 + warp * 128;
          double n16d = static_cast<double>(sm.n16f[v]);
          double rs = 0.0;
          for (int q = 0; q < 4; ++q) {
            const int i = lane + 32 * q;
            double y64 = 0.0;
            for (int k = 0; k < 128; ++k) y64 = fma(a.tab.pi64[i * 128 + k], static_cast<double>(sm.xt[k * kXS + v]), y64);
            const GroupBook& gb = L.g[i < L.split ? 0 : 1];
            double rr = y64 - (n16d * inv_sqrt_d64) * gb.c64[sm.codes[v * 128 + i]];
            r64[i] = rr;
            rs = fma(rr, rr, rs);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
          __syncwarp();
          for (int q = 0; q < a.m / 32; ++q) {
            const int p = lane + 32 * q;
            double zz = 0.0;
            for (int j = 0; j < 128; ++j) zz = fma(a.tab.s64[p * 128 + j], r64[j], zz);
            unsigned w = __ballot_sync(0xffffffffu, zz >= 0.0);
            if (lane == 0) sm.sword[v * 4 + q] = w;
          }
          r16 = __half_as_ushort(__double2half(sqrt(rs)));
          if (lane == 0) atomicAdd(&a.tab.counters[1], 1ULL);
          __syncwarp();
        } else {
          r16 = __half_as_ushort(__float2half_rn(sqrtf(sm.rho2[v])));
        }
      }
      const int pos = a.start_pos[b] + t;
      const int blk = pos >> 4;
      if (pos < 0 || blk >= a.maxp) {
        if (lane == 0) atomicOr(a.tab.err, kErrBlock);
        continue;
      }
      const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) atomicOr(a.tab.err, kErrPage);
        continue;
      }
      const int slot = pos & 15;
      unsigned char* base = a.cache + static_cast<long long>(page) * a.page_bytes +
                            static_cast<long long>(h) * L.block_bytes;
      const int nwords = L.code_bytes / 4;
      for (int w = lane; w < nwords; w += 32) {
        reinterpret_cast<unsigned*>(base + slot * L.code_bytes)[w] = pack_code_word(L, sm.codes + v * 128, w);
      }
      if (KEY && L.qjl) {
        const int sw = a.m / 32;
        if (lane < sw) {
          unsigned word;
          if (refine) {
            word = sm.sword[v * 4 + lane];
          } else {
            word = 0;
            for (int l = 0; l < 8; ++l) word |= static_cast<unsigned>(sm.snib[v * 32 + 8 * lane + l]) << (4 * l);
          }
          reinterpret_cast<unsigned*>(base + L.off_signs + slot * (a.m / 8))[lane] = word;
        }
        if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_rnorm)[slot] = r16;
      }
      if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_norm)[slot] = sm.n16[v];
    }
    __syncthreads();
  }
}

template <bool KEY>
cudaError_t launch_kind(const QuantizeArgs& a, cudaStream_t s) {
  static std::atomic<unsigned long long> configured{0};
  const size_t smem = smem_bytes<KEY>();
  const cudaError_t e = smem_attr_once(quantize_kernel<KEY>, static_cast<int>(smem), configured);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  const long long ntiles = (nvec + kTile - 1) / kTile;
  const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
  quantize_kernel<KEY><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_impl(const QuantizeArgs& a, cudaStream_t s) {
  if (a.lay.qjl) return launch_kind<true>(a, s);
  return launch_kind<false>(a, s);
}

// ---------------------------------------------------------------------------
// Latency-first append of a few vectors (a decode step's new token per
// sequence and KV head): one warp per vector, four vectors per CTA (each warp
// reads all of Pi^T from shared memory: few warps per SM keep that short), K
// and V vectors in one launch (CTAs [0, nbk) keys, the rest values).  Pi^T
// (and for keys S^T) are staged once per CTA by asynchronous 16-byte copies,
// all in flight at once; the fast
// path is the tile kernel's above, vector by vector: y = Pi x summed over k in
// order (fp32), the same code and sign guards, the same packing.  A decision
// inside a guard is retaken in fp64 by the whole warp, one decision at a time
// (a lane takes four of the 128 terms, so each costs one round of loads):
// a code from y_j = Pi_j x, a sign bit from z_p = (S Pi)_p x - fp16(||x||) /
// sqrt(d) S_p c^ (the product S Pi as a double-float table, the codes as
// decided).  The residual norm stays the fp32 one.  Lane l holds channels
// (projections) 4 l .. 4 l + 3.
constexpr int kAppWarps = 4;
constexpr int kAppScratch = 128 * 4 + 128 * 4 + 128;   // x, r, codes per warp
constexpr int kAppSmem = 2 * 128 * 128 * 4 + kAppWarps * kAppScratch;

__device__ void append_vector(const QuantizeArgs& a, bool key, long long gv, const float* pit, const float* st,
                              unsigned char* scratch, int lane) {
  const KindLayout& L = a.lay;
  float* xs = reinterpret_cast<float*>(scratch);
  float* rs = xs + 128;
  unsigned char* codes = reinterpret_cast<unsigned char*>(rs + 128);
  const float inv_sqrt_d = 0.08838834764831845f;
  const double inv_sqrt_d64 = 1.0 / sqrt(128.0);
  const double sqrt_d64 = sqrt(128.0);
  // 1. x and its double-float squared norm
  float xv[4];
  if (a.f32) {
    const float4 x4 = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + gv * kD)[lane];
    xv[0] = x4.x, xv[1] = x4.y, xv[2] = x4.z, xv[3] = x4.w;
  } else {
    const uint2 x2 = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.x) + gv * kD)[lane];
    xv[0] = __uint_as_float(x2.x << 16), xv[1] = __uint_as_float(x2.x & 0xFFFF0000u);
    xv[2] = __uint_as_float(x2.y << 16), xv[3] = __uint_as_float(x2.y & 0xFFFF0000u);
  }
  *reinterpret_cast<float4*>(xs + 4 * lane) = make_float4(xv[0], xv[1], xv[2], xv[3]);
  float sh = 0.0f, sl = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float p = xv[q] * xv[q];
    const float e = fmaf(xv[q], xv[q], -p);
    float s, t;
    two_sum(sh, p, s, t);
    sh = s;
    sl += t + e;
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float bh = __shfl_xor_sync(0xffffffffu, sh, o), bl = __shfl_xor_sync(0xffffffffu, sl, o);
    df_add(sh, sl, bh, bl);
  }
  float nh = 0.0f, nl = 0.0f;
  if (sh > 0.0f) {
    const float r = sqrtf(sh);
    const float res = fmaf(-r, r, sh) + sl;
    fast_two_sum(r, res / (2.0f * r), nh, nl);
  }
  const float scale = nh > 0.0f ? 11.313708498984761f / nh : 0.0f;   // sqrt(128) / ||x||
  const __half n16 = df_to_half(nh, nl);
  const float n16f = __half2float(n16);
  __syncwarp();
  // 2. y = Pi x for outputs 4 lane .. 4 lane + 3
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int k = 0; k < 128; ++k) {
    const float4 p = *reinterpret_cast<const float4*>(pit + k * 128 + 4 * lane);
    const float xk = xs[k];
    y[0] = fmaf(p.x, xk, y[0]);
    y[1] = fmaf(p.y, xk, y[1]);
    y[2] = fmaf(p.z, xk, y[2]);
    y[3] = fmaf(p.w, xk, y[3]);
  }
  // 3. codes (fp64 re-decision near a boundary); keys: the residual
  float rpart = 0.0f;
  unsigned cw = 0;
  int code4[4];
  unsigned guarded = 0;          // bit oi: channel 4 lane + oi within the code guard
#pragma unroll
  for (int oi = 0; oi < 4; ++oi) {
    const int i = 4 * lane + oi;
    const GroupBook& gb = L.g[i < L.split ? 0 : 1];
    const float u = y[oi] * scale;
    int code = 0;
    float mind = INFINITY;
    for (int k = 0; k < gb.nb; ++k) {
      code += u >= gb.t[k];
      mind = fminf(mind, fabsf(u - gb.t[k]));
    }
    code4[oi] = code;
    if (mind < kCodeGuard) guarded |= 1u << oi;
  }
  // the guarded codes in fp64, the warp together on each
  const double n64 = static_cast<double>(nh) + static_cast<double>(nl);
#pragma unroll
  for (int oi = 0; oi < 4; ++oi) {
    unsigned todo = __ballot_sync(0xffffffffu, (guarded >> oi) & 1u);
    while (todo) {
      const int src = __ffs(todo) - 1;
      todo &= todo - 1u;
      const int i = 4 * src + oi;
      const double2 p0 = *reinterpret_cast<const double2*>(a.tab.pi64 + i * 128 + 4 * lane);
      const double2 p1 = *reinterpret_cast<const double2*>(a.tab.pi64 + i * 128 + 4 * lane + 2);
      double y64 = fma(p0.x, static_cast<double>(xs[4 * lane]), fma(p0.y, static_cast<double>(xs[4 * lane + 1]),
                   fma(p1.x, static_cast<double>(xs[4 * lane + 2]), p1.y * static_cast<double>(xs[4 * lane + 3]))));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) y64 += __shfl_xor_sync(0xffffffffu, y64, o);
      if (lane == src) {
        const GroupBook& gb = L.g[i < L.split ? 0 : 1];
        const double u64 = n64 > 0.0 ? sqrt_d64 * y64 / n64 : 0.0;
        int code = 0;
        for (int k = 0; k < gb.nb; ++k) code += u64 >= gb.t64[k];
        code4[oi] = code;
        atomicAdd(&a.tab.counters[0], 1ULL);
      }
    }
  }
#pragma unroll
  for (int oi = 0; oi < 4; ++oi) {
    const int i = 4 * lane + oi;
    const GroupBook& gb = L.g[i < L.split ? 0 : 1];
    const int code = code4[oi];
    cw |= static_cast<unsigned>(code) << (8 * oi);
    if (key) {
      const float r = fmaf(-n16f * inv_sqrt_d, gb.c[code], y[oi]);
      rs[i] = r;
      rpart = fmaf(r, r, rpart);
    }
  }
  *reinterpret_cast<unsigned*>(codes + 4 * lane) = cw;
  unsigned sword = 0;          // lanes 0 .. m/32 - 1: sign word `lane`
  bool refine = false;
  float rho2 = 0.0f;
  if (key && L.qjl) {
    rho2 = rpart;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rho2 += __shfl_xor_sync(0xffffffffu, rho2, o);
    __syncwarp();
    // 4. z = S r for projections 4 lane .. 4 lane + 3
    float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int j = 0; j < 128; ++j) {
      const float4 s4 = *reinterpret_cast<const float4*>(st + j * 128 + 4 * lane);
      const float rj = rs[j];
      z[0] = fmaf(s4.x, rj, z[0]);
      z[1] = fmaf(s4.y, rj, z[1]);
      z[2] = fmaf(s4.z, rj, z[2]);
      z[3] = fmaf(s4.w, rj, z[3]);
    }
    const float guard = kSignGuard * sqrtf(rho2);
    unsigned nib = 0, near = 0;
#pragma unroll
    for (int oi = 0; oi < 4; ++oi) {
      nib |= (z[oi] >= 0.0f ? 1u : 0u) << oi;
      if (4 * lane + oi < a.m && fabsf(z[oi]) < guard) near |= 1u << oi;
    }
    // word w = projections 32 w .. 32 w + 31 = the nibbles of lanes 8 w .. 8 w + 7
#pragma unroll
    for (int l = 0; l < 8; ++l) {
      const unsigned n = __shfl_sync(0xffffffffu, nib, (8 * lane + l) & 31);
      sword |= n << (4 * l);
    }
    // the guarded sign bits in fp64: z_p = (S Pi)_p x - n16 / sqrt(d) S_p c^, the warp together on each;
    // lane l's terms are channels 4 l .. 4 l + 3 (their codes are this lane's)
    const double ns = static_cast<double>(n16f) * inv_sqrt_d64;
    double cx[4], xd[4];
#pragma unroll
    for (int oi = 0; oi < 4; ++oi) {
      const int j = 4 * lane + oi;
      cx[oi] = ns * L.g[j < L.split ? 0 : 1].c64[code4[oi]];
      xd[oi] = static_cast<double>(xs[j]);
    }
#pragma unroll
    for (int oi = 0; oi < 4; ++oi) {
      unsigned todo = __ballot_sync(0xffffffffu, (near >> oi) & 1u);
      if (todo) refine = true;
      while (todo) {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int pj = 4 * src + oi;
        const float4 a0 = *reinterpret_cast<const float4*>(a.tab.a_df + (pj * 128 + 4 * lane) * 2);
        const float4 a1 = *reinterpret_cast<const float4*>(a.tab.a_df + (pj * 128 + 4 * lane) * 2 + 4);
        const double2 s0 = *reinterpret_cast<const double2*>(a.tab.s64 + pj * 128 + 4 * lane);
        const double2 s1 = *reinterpret_cast<const double2*>(a.tab.s64 + pj * 128 + 4 * lane + 2);
        double zz = fma(static_cast<double>(a0.x) + static_cast<double>(a0.y), xd[0], -s0.x * cx[0]);
        zz += fma(static_cast<double>(a0.z) + static_cast<double>(a0.w), xd[1], -s0.y * cx[1]);
        zz += fma(static_cast<double>(a1.x) + static_cast<double>(a1.y), xd[2], -s1.x * cx[2]);
        zz += fma(static_cast<double>(a1.z) + static_cast<double>(a1.w), xd[3], -s1.y * cx[3]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) zz += __shfl_xor_sync(0xffffffffu, zz, o);
        if (lane == (pj >> 5)) sword = (sword & ~(1u << (pj & 31))) | ((zz >= 0.0 ? 1u : 0u) << (pj & 31));
      }
    }
  }
  unsigned short r16 = 0;
  if (key && L.qjl) {
    r16 = __half_as_ushort(__float2half_rn(sqrtf(rho2)));
    if (refine && lane == 0) atomicAdd(&a.tab.counters[1], 1ULL);
  }
  __syncwarp();
  // 5. store at (page, slot, head)
  const int h = static_cast<int>(gv % a.H);
  const long long bt = gv / a.H;
  const int t = static_cast<int>(bt % a.n_new);
  const int b = static_cast<int>(bt / a.n_new);
  const int pos = a.start_pos[b] + t;
  const int blk = pos >> 4;
  if (pos < 0 || blk >= a.maxp) {
    if (lane == 0) atomicOr(a.tab.err, kErrBlock);
    return;
  }
  const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) atomicOr(a.tab.err, kErrPage);
    return;
  }
  const int slot = pos & 15;
  unsigned char* base = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(h) * L.block_bytes;
  for (int w = lane; w < L.code_bytes / 4; w += 32)
    reinterpret_cast<unsigned*>(base + slot * L.code_bytes)[w] = pack_code_word(L, codes, w);
  if (key && L.qjl) {
    if (lane < a.m / 32) reinterpret_cast<unsigned*>(base + L.off_signs + slot * (a.m / 8))[lane] = sword;
    if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_rnorm)[slot] = r16;
  }
  if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_norm)[slot] = __half_as_ushort(n16);
}

__global__ void __launch_bounds__(32 * kAppWarps, 1) append_kernel(QuantizeArgs ka, QuantizeArgs va, int nbk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* pit = reinterpret_cast<float*>(smem_raw);
  float* st = pit + 128 * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool key = static_cast<int>(blockIdx.x) < nbk;
  const QuantizeArgs& a = key ? ka : va;
  const bool qjl = key && a.lay.qjl;
  pdl_trigger();                       // the query prep may start now (it waits for this grid before it ends)
  // the matrices: every 16-byte copy of the CTA in flight at once
  {
    const uint32_t pit_s = static_cast<uint32_t>(__cvta_generic_to_shared(pit));
    const uint32_t st_s = static_cast<uint32_t>(__cvta_generic_to_shared(st));
    for (int v = tid; v < 128 * 128 / 4; v += 32 * kAppWarps)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(pit_s + 16 * v), "l"(a.tab.pit + 4 * v) : "memory");
    if (qjl) {
      // S^T with rows of m projections, as [128][128] (projections >= m zero-filled)
      for (int v = tid; v < 128 * 128 / 4; v += 32 * kAppWarps) {
        const int j = v >> 5, c = 4 * (v & 31);
        const float* src = a.tab.st + j * a.m + (c < a.m ? c : 0);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(st_s + 16 * v), "l"(src),
                     "r"(c < a.m ? 16 : 0) : "memory");
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }
  __syncthreads();
  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  const long long gv = static_cast<long long>(key ? blockIdx.x : blockIdx.x - nbk) * kAppWarps + warp;
  if (gv < nvec)
    append_vector(a, key, gv, pit, st, smem_raw + 2 * 128 * 128 * 4 + warp * kAppScratch, lane);
}

}  // namespace

// Supported: d = 128, m a multiple of 32 (at most 128), 16-byte aligned inputs;
// at most 2^16 CTAs.  False: the caller takes another quantize kernel.
cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s) { return launch_quantize_impl(a, s); }

bool launch_append(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err) {
  const QuantizeArgs& a0 = k.x ? k : v;
  if (!k.x && !v.x) return false;
  if (k.x && k.lay.qjl && (k.m % 32 || k.m > 128 || k.m < 32)) return false;
  const long long nvec = static_cast<long long>(a0.batch) * a0.n_new * a0.H;
  const long long nb = (nvec + kAppWarps - 1) / kAppWarps;
  const long long nbk = k.x ? nb : 0, nbv = v.x ? nb : 0;
  if (nbk + nbv > 65535) return false;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = smem_attr_once(append_kernel, kAppSmem, configured);
  if (e == cudaSuccess) {
    append_kernel<<<static_cast<unsigned>(nbk + nbv), 32 * kAppWarps, kAppSmem, s>>>(k, v, static_cast<int>(nbk));
    e = cudaGetLastError();
  }
  *err = e;
  return true;
}

}  // namespace tq
