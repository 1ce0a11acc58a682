// Quantize and decode attention for head dimensions other than 128 (d a
// multiple of 32, at most 256): plain CUDA-core kernels for any bit widths and
// splits; the tensor-core and lookup-table kernels serve d = 128.
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §4.2: the codebook is
// fitted once per (d, b); §4.1 rotation, §4.3 residual + QJL; §2.2 decode;
// [P2] "생각정리 209 (TurboQuant)", stages 1-2.
//
// quantize: a warp takes four vectors; lanes own output channels j = lane + 32 i.
//   y = Pi x in fp32 (Pi^T rows read across the lanes); u = sqrt(d) y / ||x||,
//   code = #{k : u >= t_k}; a u within 2e-5 of a boundary is decided again in
//   fp64 (y_j and ||x|| recomputed).  Keys: r = y - fp16(||x||)/sqrt(d) c[code],
//   z = S r in fp32 (S^T rows across the lanes); when some |z_p| < 5e-5 ||r||
//   the vector's y, r and those z_p are recomputed in fp64.  The fp16 norm is
//   exactly rounded (fp64 when the fp32 norm lies within 1e-5 of a midpoint).
// decode: qprep (one block per query row, W = [Pi; S Pi] columns across the
//   threads), partials (one block of eight warps per (sequence, KV head, chunk);
//   a warp takes one token at a time, lanes own d/32 channels and m/32
//   projections, online softmax per query head; the warps' states are merged
//   in shared memory), merge (log-sum-exp over the chunks, o = Pi^T (acc / l)).

#include "tq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

constexpr int kGDMax = 256;          // largest head dimension
constexpr int kGQVecs = 4;           // vectors per warp (quantize)
constexpr int kGQWarps = 4;          // warps per quantize block
constexpr float kGCodeGuard = 2e-5f;
constexpr float kGSignGuard = 5e-5f;
constexpr float kSqrtHalfPiG = 1.2533141373155003f;

__device__ __forceinline__ float gwarp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double gwarp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float gwarp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float load_x(const void* x, bool f32, long long idx) {
  return f32 ? static_cast<const float*>(x)[idx] : __bfloat162float(static_cast<const __nv_bfloat16*>(x)[idx]);
}

// Stored value of a code (tq.h): 4-bit fields are sign-magnitude.
__device__ __forceinline__ uint32_t stored_value(int b, int code) {
  return b == 4 ? static_cast<uint32_t>(code >= 8 ? code - 8 : 15 - code) : static_cast<uint32_t>(code);
}
// OR the code of channel j into a record's code words (shared memory; lanes
// sharing a word use atomics).
__device__ void put_code_generic(uint32_t* words, const KindLayout& L, int j, int code) {
  const int grp = j < L.split ? 0 : 1, b = L.g[grp].bits, c = grp ? j - L.split : j;
  const int base = grp ? L.split * L.g[0].bits : 0;
  if (b == 3) {
    const int ob = base + 24 * (c >> 3), i = c & 7;
    if (i < 6) {
      const int pos = ob + 4 * i;
      atomicOr(words + (pos >> 5), static_cast<uint32_t>(code) << (pos & 31));
    } else {
      for (int q = 0; q < 3; ++q) {
        const int pos = ob + 3 + 4 * (i - 6) + 8 * q;
        atomicOr(words + (pos >> 5), static_cast<uint32_t>((code >> q) & 1) << (pos & 31));
      }
    }
    return;
  }
  const int pos = base + b * c;
  atomicOr(words + (pos >> 5), stored_value(b, code) << (pos & 31));
}
// Code of channel j from a record's code words (any format).
__device__ int get_code_generic(const uint32_t* w, int bh, int bl, int split, int j) {
  const int grp = j < split ? 0 : 1, b = grp ? bl : bh, c = grp ? j - split : j, base = grp ? split * bh : 0;
  auto bitsat = [&](int off, int n) { return static_cast<int>((w[off >> 5] >> (off & 31)) & ((1u << n) - 1u)); };
  if (b == 3) {
    const int ob = base + 24 * (c >> 3), i = c & 7;
    if (i < 6) return bitsat(ob + 4 * i, 3);
    const int s0 = ob + 3 + 4 * (i - 6);
    return bitsat(s0, 1) | (bitsat(s0 + 8, 1) << 1) | (bitsat(s0 + 16, 1) << 2);
  }
  const int v = bitsat(base + b * c, b);
  if (b == 4) return (v & 8) ? 7 - (v & 7) : 8 + v;
  return v;
}

// ---------------------------------------------------------------------------
// quantize
// ---------------------------------------------------------------------------
struct GenQArgs {
  QuantizeArgs q;
  int d;
};

__global__ void __launch_bounds__(32 * kGQWarps) generic_quantize_kernel(GenQArgs ga) {
  const QuantizeArgs& a = ga.q;
  const int d = ga.d, nj = d / 32, m = a.m;
  const bool key = a.lay.qjl != 0;
  __shared__ float xs[kGQWarps][kGQVecs][kGDMax];
  __shared__ float rs[kGQWarps][kGQVecs][kGDMax];
  __shared__ uint32_t cwords[kGQWarps][kGQVecs][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  const long long v0 = (static_cast<long long>(blockIdx.x) * kGQWarps + warp) * kGQVecs;
  if (v0 >= nvec) return;
  const float sqrt_d = sqrtf(static_cast<float>(d));
  const double sqrt_d64 = sqrt(static_cast<double>(d));

  // x, norms, record locations
  float nf[kGQVecs];
  __half n16[kGQVecs];
  unsigned char* rec[kGQVecs];
  int slot[kGQVecs];
#pragma unroll
  for (int v = 0; v < kGQVecs; ++v) {
    const long long gv = v0 + v;
    const bool ok = gv < nvec;
    float ss = 0.0f;
    for (int i = 0; i < nj; ++i) {
      const int k = lane + 32 * i;
      const float xv = ok ? load_x(a.x, a.f32, gv * d + k) : 0.0f;
      xs[warp][v][k] = xv;
      ss = fmaf(xv, xv, ss);
    }
    ss = gwarp_sum(ss);
    nf[v] = ss > 0.0f ? sqrtf(ss) : 0.0f;
    n16[v] = __float2half_rn(nf[v]);
    // an fp32 norm near an fp16 rounding midpoint: the fp64 norm decides
    bool near = false;
    if (nf[v] > 0.0f) {
      const float hb = __half2float(n16[v]);
      const unsigned short hbits = __half_as_ushort(n16[v]);
      const float up = __half2float(__ushort_as_half(static_cast<unsigned short>(hbits + 1)));
      const float dn = hbits ? __half2float(__ushort_as_half(static_cast<unsigned short>(hbits - 1))) : 0.0f;
      near = fabsf(nf[v] - 0.5f * (hb + up)) < 1e-5f * nf[v] || fabsf(nf[v] - 0.5f * (hb + dn)) < 1e-5f * nf[v];
    }
    if (near) {          // warp-uniform (nf is the same in every lane)
      double s64 = 0.0;
      for (int i = 0; i < nj; ++i) {
        const double xv = xs[warp][v][lane + 32 * i];
        s64 = fma(xv, xv, s64);
      }
      s64 = gwarp_sum_d(s64);
      n16[v] = __double2half(sqrt(s64));
    }
    cwords[warp][v][lane] = 0u;
    rec[v] = nullptr;
    slot[v] = 0;
    if (ok) {
      const long long bt = gv / a.H;
      const int hh = static_cast<int>(gv % a.H), t = static_cast<int>(bt % a.n_new), b = static_cast<int>(bt / a.n_new);
      const int pos = a.start_pos[b] + t, blk = pos >> 4;
      if (pos < 0 || blk >= a.maxp) {
        if (lane == 0) atomicOr(a.tab.err, kErrBlock);
      } else {
        const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
        if (page < 0 || page >= a.num_pages) {
          if (lane == 0) atomicOr(a.tab.err, kErrPage);
        } else {
          rec[v] = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(hh) * a.lay.block_bytes;
          slot[v] = pos & 15;
        }
      }
    }
  }
  __syncwarp();

  // y = Pi x (fp32): lane owns y_j, j = lane + 32 i; Pi^T row k is contiguous in j
  float y[kGQVecs][kGDMax / 32];
#pragma unroll
  for (int v = 0; v < kGQVecs; ++v)
#pragma unroll
    for (int i = 0; i < kGDMax / 32; ++i) y[v][i] = 0.0f;
  for (int k = 0; k < d; ++k) {
    float pk[kGDMax / 32];
#pragma unroll
    for (int i = 0; i < kGDMax / 32; ++i) pk[i] = i < nj ? __ldg(a.tab.pit + static_cast<long long>(k) * d + lane + 32 * i) : 0.0f;
#pragma unroll
    for (int v = 0; v < kGQVecs; ++v) {
      const float xk = xs[warp][v][k];
#pragma unroll
      for (int i = 0; i < kGDMax / 32; ++i) y[v][i] = fmaf(pk[i], xk, y[v][i]);
    }
  }

#pragma unroll
  for (int v = 0; v < kGQVecs; ++v) {
    const long long gv = v0 + v;
    if (gv >= nvec) break;                       // warp-uniform
    const float n16f = __half2float(n16[v]);
    const float ku = nf[v] > 0.0f ? sqrt_d / nf[v] : 0.0f;
    double n64 = -1.0;                           // exact norm, computed when first needed
    float rho2 = 0.0f;
    for (int i = 0; i < nj; ++i) {
      const int j = lane + 32 * i;
      const int grp = j < a.lay.split ? 0 : 1;
      const GroupBook& gb = a.lay.g[grp];
      const float u = y[v][i] * ku;
      int code = 0;
      float dmin = INFINITY;
      for (int k = 0; k < gb.nb; ++k) {
        code += u >= gb.t[k] ? 1 : 0;
        dmin = fminf(dmin, fabsf(u - gb.t[k]));
      }
      if (dmin < kGCodeGuard && nf[v] > 0.0f) {   // rare: decide in fp64 (this lane alone)
        if (n64 < 0.0) {
          double s64 = 0.0;
          for (int k = 0; k < d; ++k) s64 = fma(static_cast<double>(xs[warp][v][k]), xs[warp][v][k], s64);
          n64 = sqrt(s64);
        }
        double y64 = 0.0;
        for (int k = 0; k < d; ++k) y64 = fma(a.tab.pi64[static_cast<long long>(j) * d + k], xs[warp][v][k], y64);
        const double u64 = sqrt_d64 * y64 / n64;
        code = 0;
        for (int k = 0; k < gb.nb; ++k) code += u64 >= gb.t64[k] ? 1 : 0;
        atomicAdd(&a.tab.counters[0], 1ULL);
      }
      put_code_generic(cwords[warp][v], a.lay, j, code);
      if (key) {
        // zero fp16 norm: the residual is y itself (its signs are those of S y)
        const float r = n16f > 0.0f ? y[v][i] - n16f / sqrt_d * gb.c[code] : y[v][i];
        rs[warp][v][j] = r;
        rho2 = fmaf(r, r, rho2);
      }
    }
    __syncwarp();
    unsigned char* rc = rec[v];
    if (rc) {
      const int cw = a.lay.code_bytes / 4;
      uint32_t* dst = reinterpret_cast<uint32_t*>(rc + slot[v] * a.lay.code_bytes);
      for (int w = lane; w < cw; w += 32) dst[w] = cwords[warp][v][w];
      if (lane == 0) *(reinterpret_cast<unsigned short*>(rc + a.lay.off_norm) + slot[v]) = __half_as_ushort(n16[v]);
    }
    if (!key) continue;
    rho2 = gwarp_sum(rho2);
    const float rho = sqrtf(rho2);
    // z = S r: lane owns z_p, p = lane + 32 i; S^T row j is contiguous in p
    const int np = m / 32;
    float z[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < d; ++j) {
      const float rj = rs[warp][v][j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < np) z[i] = fmaf(__ldg(a.tab.st + static_cast<long long>(j) * m + lane + 32 * i), rj, z[i]);
    }
    bool flag = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < np && fabsf(z[i]) < kGSignGuard * rho) flag = true;
    if (__any_sync(0xffffffffu, flag)) {
      // rare: this vector's residual and the flagged projections in fp64
      if (n64 < 0.0) {
        double s64 = 0.0;
        for (int k = 0; k < d; ++k) s64 = fma(static_cast<double>(xs[warp][v][k]), xs[warp][v][k], s64);
        n64 = sqrt(s64);
      }
      __shared__ double r64s[kGQWarps][kGDMax];
      for (int i = 0; i < nj; ++i) {
        const int j = lane + 32 * i;
        double y64 = 0.0;
        for (int k = 0; k < d; ++k) y64 = fma(a.tab.pi64[static_cast<long long>(j) * d + k], xs[warp][v][k], y64);
        const int code = get_code_generic(cwords[warp][v], a.lay.g[0].bits, a.lay.g[1].bits, a.lay.split, j);
        const int grp = j < a.lay.split ? 0 : 1;
        r64s[warp][j] = n16f > 0.0f ? y64 - static_cast<double>(n16f) / sqrt_d64 * a.lay.g[grp].c64[code] : y64;
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < np && fabsf(z[i]) < kGSignGuard * rho) {
          const int p = lane + 32 * i;
          double z64 = 0.0;
          for (int j = 0; j < d; ++j) z64 = fma(a.tab.s64[static_cast<long long>(p) * d + j], r64s[warp][j], z64);
          z[i] = z64 >= 0.0 ? 1.0f : -1.0f;
          atomicAdd(&a.tab.counters[1], 1ULL);
        }
      }
      __syncwarp();
    }
    if (rc) {
      uint32_t* sg = reinterpret_cast<uint32_t*>(rc + a.lay.off_signs + slot[v] * (m / 8));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < np) {
          const uint32_t word = __ballot_sync(0xffffffffu, z[i] >= 0.0f);   // bit = projection 32 i + lane
          if (lane == 0) sg[i] = word;
        }
      }
      if (lane == 0)
        *(reinterpret_cast<unsigned short*>(rc + a.lay.off_rnorm) + slot[v]) =
            __half_as_ushort(__float2half_rn(rho));
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
struct GenDArgs {
  DecodeArgs a;
  int d;
};

// [q~; u] = W q, one block per query row, thread r computes output r.
__global__ void generic_qprep_kernel(GenDArgs ga) {
  const DecodeArgs& a = ga.a;
  const int d = ga.d, nout = d + a.m;
  __shared__ float qs[kGDMax];
  const long long row = blockIdx.x;
  for (int k = threadIdx.x; k < d; k += blockDim.x) qs[k] = load_x(a.q, a.f32, row * d + k);
  __syncthreads();
  for (int r = threadIdx.x; r < nout; r += blockDim.x) {
    float acc = 0.0f;
    for (int k = 0; k < d; ++k) acc = fmaf(__ldg(a.tab.wt + static_cast<long long>(k) * nout + r), qs[k], acc);
    a.qprep[row * nout + r] = acc;
  }
}

constexpr int kGPWarps = 8;

// Partials of one (chunk, KV head, sequence): running max, sum and value
// accumulator per query head of the group, [row][chunk][d + 2].
__global__ void __launch_bounds__(32 * kGPWarps) generic_partials_kernel(GenDArgs ga) {
  const DecodeArgs& a = ga.a;
  const int d = ga.d, m = a.m, nout = d + m, G = a.G, nj = d / 32, np = m / 32;
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  extern __shared__ float gsm[];
  float* qv = gsm;                               // [G][nout]: q~ then u
  float* mst = qv + G * nout;                    // [G] merged state: max
  float* lst = mst + kMaxGroup;                  // [G] sum
  float* ast = lst + kMaxGroup;                  // [G][d] accumulator
  for (int idx = threadIdx.x; idx < G * nout; idx += blockDim.x) {
    const int g = idx / nout, r = idx % nout;
    qv[idx] = a.qprep[(static_cast<long long>(b) * a.Hq + h * G + g) * nout + r];
  }
  int L = a.seq_lens[b] + a.len_add;
  if (L < 0 || L > a.max_seq_len || L > a.maxp * kPage) {
    if (threadIdx.x == 0 && chunk == 0 && h == 0) atomicOr(a.tab.err, kErrSeqLen);
    L = max(0, min(L, min(a.max_seq_len, a.maxp * kPage)));
  }
  __syncthreads();
  const int t0 = chunk * a.chunk, t1 = min(t0 + a.chunk, L);
  const float inv_sqrt_d = rsqrtf(static_cast<float>(d));
  const float qjl = kSqrtHalfPiG / static_cast<float>(m);
  float mr[kMaxGroup], lr[kMaxGroup], acc[kMaxGroup][kGDMax / 32];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    mr[g] = -INFINITY;
    lr[g] = 0.0f;
#pragma unroll
    for (int i = 0; i < kGDMax / 32; ++i) acc[g][i] = 0.0f;
  }
  for (int t = t0 + warp; t < t1; t += kGPWarps) {
    const int page = a.block_table[static_cast<long long>(b) * a.maxp + (t >> 4)];
    if (page < 0 || page >= a.num_pages) {
      if (lane == 0) atomicOr(a.tab.err, kErrPage);
      continue;
    }
    const int slot = t & 15;
    const unsigned char* kb = a.kc + static_cast<long long>(page) * a.k_page_bytes + static_cast<long long>(h) * a.kl.block_bytes;
    const unsigned char* vb = a.vc + static_cast<long long>(page) * a.v_page_bytes + static_cast<long long>(h) * a.vl.block_bytes;
    const uint32_t* kw = reinterpret_cast<const uint32_t*>(kb + slot * a.kl.code_bytes);
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(vb + slot * a.vl.code_bytes);
    float s1[kMaxGroup], s2[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) s1[g] = s2[g] = 0.0f;
    for (int i = 0; i < nj; ++i) {
      const int j = lane + 32 * i;
      const float c = a.kl.g[j < a.kl.split ? 0 : 1].c[get_code_generic(kw, a.kl.g[0].bits, a.kl.g[1].bits, a.kl.split, j)];
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g)
        if (g < G) s1[g] = fmaf(c, qv[g * nout + j], s1[g]);
    }
    if (a.kl.qjl) {
      const uint32_t* sw = reinterpret_cast<const uint32_t*>(kb + a.kl.off_signs + slot * (m / 8));
      for (int i = 0; i < np; ++i) {
        const bool pos = (sw[i] >> lane) & 1u;
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g)
          if (g < G) {
            const float u = qv[g * nout + d + 32 * i + lane];
            s2[g] += pos ? u : -u;
          }
      }
    }
    const float nk = __half2float(reinterpret_cast<const __half*>(kb + a.kl.off_norm)[slot]);
    const float rk = a.kl.qjl ? __half2float(reinterpret_cast<const __half*>(kb + a.kl.off_rnorm)[slot]) : 0.0f;
    const float nv = __half2float(reinterpret_cast<const __half*>(vb + a.vl.off_norm)[slot]) * inv_sqrt_d;
    float cv[kGDMax / 32];
#pragma unroll
    for (int i = 0; i < kGDMax / 32; ++i) {
      const int j = lane + 32 * i;
      cv[i] = i < nj ? a.vl.g[j < a.vl.split ? 0 : 1].c[get_code_generic(vw, a.vl.g[0].bits, a.vl.g[1].bits, a.vl.split, j)]
                     : 0.0f;
    }
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      const float lg = (nk * inv_sqrt_d * gwarp_sum(s1[g]) + qjl * rk * gwarp_sum(s2[g])) * a.scale_log2;
      const float mn = fmaxf(mr[g], lg);
      const float al = exp2f(mr[g] - mn), p = exp2f(lg - mn);
      lr[g] = lr[g] * al + p;
      mr[g] = mn;
#pragma unroll
      for (int i = 0; i < kGDMax / 32; ++i) acc[g][i] = fmaf(p * nv, cv[i], acc[g][i] * al);
    }
  }
  // merge the warps' states, one warp at a time
  for (int w = 0; w < kGPWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g >= G) break;
        const float mo = w == 0 ? -INFINITY : mst[g];
        const float mn = fmaxf(mo, mr[g]);
        const float ao = mn == -INFINITY ? 0.0f : exp2f(mo - mn), an = mn == -INFINITY ? 0.0f : exp2f(mr[g] - mn);
        __syncwarp();
        if (lane == 0) {
          lst[g] = (w == 0 ? 0.0f : lst[g]) * ao + lr[g] * an;
          mst[g] = mn;
        }
#pragma unroll
        for (int i = 0; i < kGDMax / 32; ++i)
          if (i < nj) {
            const int j = lane + 32 * i;
            ast[g * d + j] = (w == 0 ? 0.0f : ast[g * d + j]) * ao + acc[g][i] * an;
          }
      }
    }
    __syncthreads();
  }
  const int nch = a.nchunks;
  for (int idx = threadIdx.x; idx < G * (d + 2); idx += blockDim.x) {
    const int g = idx / (d + 2), c = idx % (d + 2);
    const long long row = static_cast<long long>(b) * a.Hq + h * G + g;
    float* dst = a.part + (row * nch + chunk) * (d + 2);
    dst[c] = c == 0 ? mst[g] : c == 1 ? lst[g] : ast[g * d + c - 2];
  }
}

// Log-sum-exp merge of a query row's chunks and o = Pi^T (acc / l).
__global__ void generic_merge_kernel(GenDArgs ga) {
  const DecodeArgs& a = ga.a;
  const int d = ga.d;
  __shared__ float os[kGDMax];
  __shared__ float wsh[64];
  const long long row = blockIdx.x;
  int L = a.seq_lens[row / a.Hq] + a.len_add;
  L = max(0, min(L, min(a.max_seq_len, a.maxp * kPage)));
  const int nc = min(a.nchunks, (L + a.chunk - 1) / a.chunk);
  const float* P = a.part + row * a.nchunks * (d + 2);
  float M = -INFINITY;
  for (int c = 0; c < nc; ++c) M = fmaxf(M, P[static_cast<long long>(c) * (d + 2)]);
  float l = 0.0f;
  for (int c = 0; c < nc; ++c) {
    const float* pc = P + static_cast<long long>(c) * (d + 2);
    l = fmaf(pc[0] == -INFINITY ? 0.0f : exp2f(pc[0] - M), pc[1], l);
  }
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    float s = 0.0f;
    for (int c = 0; c < nc; ++c) {
      const float* pc = P + static_cast<long long>(c) * (d + 2);
      s = fmaf(pc[0] == -INFINITY ? 0.0f : exp2f(pc[0] - M), pc[2 + j], s);
    }
    os[j] = l > 0.0f ? s / l : 0.0f;
  }
  (void)wsh;
  __syncthreads();
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    float o = 0.0f;
    for (int i = 0; i < d; ++i) o = fmaf(__ldg(a.tab.pi + static_cast<long long>(i) * d + j), os[i], o);
    a.out[row * d + j] = o;
  }
}

}  // namespace

cudaError_t launch_quantize_generic(const QuantizeArgs& a, int d, cudaStream_t s) {
  const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
  if (nvec == 0) return cudaSuccess;
  const long long per_block = static_cast<long long>(kGQWarps) * kGQVecs;
  const long long blocks = (nvec + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  GenQArgs ga{a, d};
  generic_quantize_kernel<<<static_cast<unsigned>(blocks), 32 * kGQWarps, 0, s>>>(ga);
  return cudaGetLastError();
}

cudaError_t launch_decode_generic(const DecodeArgs& a, int d, int stages, cudaStream_t s) {
  GenDArgs ga{a, d};
  const long long rows = static_cast<long long>(a.B) * a.Hq;
  cudaError_t e = cudaSuccess;
  if (stages & TQ_STAGE_QPREP) {
    generic_qprep_kernel<<<static_cast<unsigned>(rows), 256, 0, s>>>(ga);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & TQ_STAGE_PARTIALS) {
    const size_t smem = sizeof(float) * (static_cast<size_t>(a.G) * (d + a.m) + 2 * kMaxGroup + kMaxGroup * d);
    generic_partials_kernel<<<dim3(a.nchunks, a.H, a.B), 32 * kGPWarps, smem, s>>>(ga);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (stages & TQ_STAGE_MERGE) {
    generic_merge_kernel<<<static_cast<unsigned>(rows), 128, 0, s>>>(ga);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace tq
