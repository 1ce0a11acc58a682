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
#include "tq_tc.cuh"

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
// (and for keys S^T) are staged once per CTA by two bulk copies while the warps
// load their vectors and norms.  The fast path is the tile kernel's above,
// vector by vector: y = Pi x summed over k in order (fp32), the same code and
// sign guards; the stored format of tq.h is built by OR-ing each code field
// into its word in shared memory.  A decision inside a guard is retaken in
// fp64 by the whole warp, one decision at a time (a lane takes four of the 128
// terms, so each costs one round of loads): a code from y_j = Pi_j x, a sign
// bit from z_p = (S Pi)_p x - fp16(||x||) / sqrt(d) S_p c^ (the product S Pi as
// a double-float table, the codes as decided).  The residual norm stays the
// fp32 one.  Lane l holds channels (projections) 4 l .. 4 l + 3.
constexpr int kAppWarps = 4;
constexpr int kAppScratch = 128 * 4 + 128 * 4 + 16 * 4;   // x, r, packed code words per warp
constexpr int kAppSmem = 2 * 128 * 128 * 4 + kAppWarps * kAppScratch;

// The kind's two codebooks, copied to shared memory once per CTA (boundaries
// past 2^b - 1 are +inf, as in GroupBook).
struct AppBook {
  float t[2][16];
  float c[2][16];
  double t64[2][16];
  double c64[2][16];
};

// Bit position of channel j's code field in the vector's code stream, the
// stored field value, and for 3-bit channels 6 and 7 of an octet the three
// single bits (see the stored format): fields never straddle a 32-bit word.
__device__ __forceinline__ void or_code(uint32_t* pw, const KindLayout& L, int bits0, int bits1, int j, int code) {
  const int g = j < L.split ? 0 : 1;
  const int b = g ? bits1 : bits0;
  const int cj = g ? j - L.split : j;
  const int base = g ? L.split * bits0 : 0;
  if (b == 3) {
    const int ob = base + 24 * (cj >> 3), i = cj & 7;
    if (i < 6) {
      const int pos = ob + 4 * i;
      atomicOr(pw + (pos >> 5), static_cast<uint32_t>(code) << (pos & 31));
    } else {
      const int s0 = ob + (i == 6 ? 3 : 7);
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int pos = s0 + 8 * q;
        atomicOr(pw + (pos >> 5), static_cast<uint32_t>((code >> q) & 1) << (pos & 31));
      }
    }
  } else {
    const uint32_t v = b == 4 ? stored4(static_cast<unsigned>(code)) : static_cast<uint32_t>(code);
    const int pos = base + b * cj;
    atomicOr(pw + (pos >> 5), v << (pos & 31));
  }
}

// Returns false when a wait for the staged matrices gave up (nothing stored).
__device__ bool append_vector(const QuantizeArgs& a, bool key, long long gv, uint32_t pit_s, uint32_t st_s,
                              const AppBook& bk, unsigned char* scratch, int lane, uint32_t bar_pi, uint32_t bar_s) {
  const KindLayout& L = a.lay;
  float* xs = reinterpret_cast<float*>(scratch);
  float* rs = xs + 128;
  uint32_t* pw = reinterpret_cast<uint32_t*>(rs + 128);
  const uint32_t xs_s = tcx::su32(xs), rs_s = tcx::su32(rs);
  const float inv_sqrt_d = 0.08838834764831845f;
  const double inv_sqrt_d64 = 1.0 / sqrt(128.0);
  const double sqrt_d64 = sqrt(128.0);
  const int g = 4 * lane < L.split ? 0 : 1;     // the group of this lane's four channels (split % 8 == 0)
  const int bits0 = L.g[0].bits, bits1 = L.g[1].bits;
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
  if (lane < 16) pw[lane] = 0u;
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
  bool failed = false;
  if (!__all_sync(0xffffffffu, tcx::bar_wait(bar_pi, 0, failed))) return false;   // Pi^T staged
  // 2. y = Pi x for outputs 4 lane .. 4 lane + 3
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 16
  for (int k = 0; k < 128; ++k) {
    const uint4 p = tcx::lds128(pit_s + 512 * k + 16 * lane);
    const float xk = tcx::ldsf(xs_s + 4 * k);
    y[0] = fmaf(__uint_as_float(p.x), xk, y[0]);
    y[1] = fmaf(__uint_as_float(p.y), xk, y[1]);
    y[2] = fmaf(__uint_as_float(p.z), xk, y[2]);
    y[3] = fmaf(__uint_as_float(p.w), xk, y[3]);
  }
  // 3. codes against the 15 boundary slots (+inf past 2^b - 1), the guarded ones
  // re-decided in fp64 by the whole warp; keys: the residual
  int code4[4] = {0, 0, 0, 0};
  unsigned guarded = 0;          // bit oi: channel 4 lane + oi within the code guard
  {
    float mind[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
    float u[4];
#pragma unroll
    for (int oi = 0; oi < 4; ++oi) u[oi] = y[oi] * scale;
#pragma unroll
    for (int k = 0; k < 15; ++k) {
      const float t = bk.t[g][k];
#pragma unroll
      for (int oi = 0; oi < 4; ++oi) {
        code4[oi] += u[oi] >= t;
        mind[oi] = fminf(mind[oi], fabsf(u[oi] - t));
      }
    }
#pragma unroll
    for (int oi = 0; oi < 4; ++oi)
      if (mind[oi] < kCodeGuard) guarded |= 1u << oi;
  }
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
      double y64 = fma(p0.x, static_cast<double>(xv[0]), fma(p0.y, static_cast<double>(xv[1]),
                   fma(p1.x, static_cast<double>(xv[2]), p1.y * static_cast<double>(xv[3]))));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) y64 += __shfl_xor_sync(0xffffffffu, y64, o);
      if (lane == src) {
        const double u64 = n64 > 0.0 ? sqrt_d64 * y64 / n64 : 0.0;
        int code = 0;
#pragma unroll
        for (int k = 0; k < 15; ++k) code += u64 >= bk.t64[g][k];
        code4[oi] = code;
        atomicAdd(&a.tab.counters[0], 1ULL);
      }
    }
  }
  float rpart = 0.0f;
#pragma unroll
  for (int oi = 0; oi < 4; ++oi) {
    or_code(pw, L, bits0, bits1, 4 * lane + oi, code4[oi]);
    if (key) {
      const float r = fmaf(-n16f * inv_sqrt_d, bk.c[g][code4[oi]], y[oi]);
      rs[4 * lane + oi] = r;
      rpart = fmaf(r, r, rpart);
    }
  }
  unsigned sword = 0;          // lanes 0 .. m/32 - 1: sign word `lane`
  bool refine = false;
  float rho2 = 0.0f;
  if (key && L.qjl) {
    rho2 = rpart;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rho2 += __shfl_xor_sync(0xffffffffu, rho2, o);
    __syncwarp();
    if (!__all_sync(0xffffffffu, tcx::bar_wait(bar_s, 0, failed))) return false;   // S^T staged
    // 4. z = S r for projections 4 lane .. 4 lane + 3 (S^T rows of m; lanes past m idle)
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t sa = st_s + 16 * (4 * lane < a.m ? lane : 0);
#pragma unroll 16
    for (int j = 0; j < 128; ++j) {
      const uint4 s4 = tcx::lds128(sa + 4 * a.m * j);
      const float rj = tcx::ldsf(rs_s + 4 * j);
      z[0] = fmaf(__uint_as_float(s4.x), rj, z[0]);
      z[1] = fmaf(__uint_as_float(s4.y), rj, z[1]);
      z[2] = fmaf(__uint_as_float(s4.z), rj, z[2]);
      z[3] = fmaf(__uint_as_float(s4.w), rj, z[3]);
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
    double cx[4];
#pragma unroll
    for (int oi = 0; oi < 4; ++oi) cx[oi] = ns * bk.c64[g][code4[oi]];
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
        double zz = fma(static_cast<double>(a0.x) + static_cast<double>(a0.y), static_cast<double>(xv[0]), -s0.x * cx[0]);
        zz += fma(static_cast<double>(a0.z) + static_cast<double>(a0.w), static_cast<double>(xv[1]), -s0.y * cx[1]);
        zz += fma(static_cast<double>(a1.x) + static_cast<double>(a1.y), static_cast<double>(xv[2]), -s1.x * cx[2]);
        zz += fma(static_cast<double>(a1.z) + static_cast<double>(a1.w), static_cast<double>(xv[3]), -s1.y * cx[3]);
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
    return true;
  }
  const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) atomicOr(a.tab.err, kErrPage);
    return true;
  }
  const int slot = pos & 15;
  unsigned char* base = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(h) * L.block_bytes;
  if (lane < L.code_bytes / 4) reinterpret_cast<unsigned*>(base + slot * L.code_bytes)[lane] = pw[lane];
  if (key && L.qjl) {
    if (lane < a.m / 32) reinterpret_cast<unsigned*>(base + L.off_signs + slot * (a.m / 8))[lane] = sword;
    if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_rnorm)[slot] = r16;
  }
  if (lane == 0) reinterpret_cast<unsigned short*>(base + L.off_norm)[slot] = __half_as_ushort(n16);
  return true;
}

__global__ void __launch_bounds__(32 * kAppWarps, 1) append_kernel(QuantizeArgs ka, QuantizeArgs va, int nbk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ AppBook bk;
  float* pit = reinterpret_cast<float*>(smem_raw);
  float* st = pit + 128 * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool key = static_cast<int>(blockIdx.x) < nbk;
  const QuantizeArgs& a = key ? ka : va;
  const bool qjl = key && a.lay.qjl;
  pdl_trigger();                       // the query prep may start now (it waits for this grid before it ends)
  // the matrices, two bulk copies (Pi^T, and S^T for keys with QJL) on their own
  // barriers: each warp takes x and its norm meanwhile, and waits for S^T only
  // when it gets to z
  __shared__ __align__(8) unsigned long long bars[2];
  const uint32_t bar_pi = tcx::su32(&bars[0]), bar_s = tcx::su32(&bars[1]);
  if (tid == 0) {
    tcx::bar_init(bar_pi, 1);
    tcx::bar_init(bar_s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tcx::bar_arrive_tx(bar_pi, 128 * 128 * 4);
    tcx::g2s(tcx::su32(pit), a.tab.pit, 128 * 128 * 4, bar_pi);
    if (qjl) {
      tcx::bar_arrive_tx(bar_s, 128 * a.m * 4);
      tcx::g2s(tcx::su32(st), a.tab.st, 128 * a.m * 4, bar_s);
    }
  }
  // the codebooks (boundaries past 2^b - 1 are +inf)
  for (int i = tid; i < 2 * 16; i += 32 * kAppWarps) {
    const int gi = i >> 4, k = i & 15;
    const GroupBook& gb = a.lay.g[gi];
    bk.t[gi][k] = k < gb.nb ? gb.t[k] : INFINITY;
    bk.t64[gi][k] = k < gb.nb ? gb.t64[k] : static_cast<double>(INFINITY);
    bk.c[gi][k] = gb.c[k];
    bk.c64[gi][k] = gb.c64[k];
  }
  __syncthreads();
  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  const long long gv = static_cast<long long>(key ? blockIdx.x : blockIdx.x - nbk) * kAppWarps + warp;
  bool ok = true;
  if (gv < nvec)
    ok = append_vector(a, key, gv, tcx::su32(pit), tcx::su32(st), bk, smem_raw + 2 * 128 * 128 * 4 + warp * kAppScratch,
                       lane, bar_pi, bar_s);
  if (!ok && lane == 0) atomicOr(a.tab.err, kErrTimeout);
  // the CTA ends only after its copies have landed (warps without a vector, or
  // a wait that gave up, may not have seen them)
  __syncthreads();
  if (tid == 0) {
    bool f = false;
    (void)tcx::bar_wait(bar_pi, 0, f);
    if (qjl) (void)tcx::bar_wait(bar_s, 0, f);
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s) { return launch_quantize_impl(a, s); }

// Supported: d = 128, m a multiple of 32 (at most 128), 16-byte aligned inputs;
// at most 2^16 CTAs.  False: the caller takes another quantize kernel.
bool launch_append(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err) {
  const QuantizeArgs& a0 = k.x ? k : v;
  if (!k.x && !v.x) return false;
  if (k.x && k.lay.qjl && (k.m % 32 || k.m > 128 || k.m < 32)) return false;
  if ((k.x && k.lay.split % 8) || (v.x && v.lay.split % 8)) return false;   // a lane's channels in one group
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
