// Online quantize-and-append on the fifth-generation tensor cores (tcgen05).
//
// [P2] "생각정리 209 (TurboQuant)", stage 1 and stage 2; [P4] riverfrot.github.io
// "TurboQuant란 무엇이며…", §4.1 (random rotation of every vector), §4.2 (the
// Lloyd-Max codebook is only looked up), §4.3 (residual r = x - Q^-1(Q(x)) and
// the 1-bit sign sketch of a random projection of r), §3.1 (paged blocks).
//
// One CTA of 16 warps per SM, persistent over tiles of 128 vectors (K tiles
// first, then V tiles, one launch).  Vector r of a tile is row r of the MMA
// and lane r of tensor memory; warp w serves lanes 32*(w%4).. (the only lanes
// it may read) and channel quarter w/4, so each vector has four threads and a
// quarter's codes fill whole 32-bit words of the record.
//   1. x rows, 16 lanes per row (8 channels each; bf16 tiles arrive in the
//      residual tile by a bulk copy issued while the previous tile was in its
//      epilogue) -> fp32 sum of squares and max by shuffles -> fp32 norm,
//      exactly rounded fp16 norm (a norm near an fp16 rounding midpoint is
//      recomputed from double-float sums of the exact squares), fp16 x scaled
//      by a power of two (exact for bf16) in a 128-byte-swizzled K-major tile.
//   2. y = x Pi^T: tcgen05.mma kind::f16, M=128 N=128, accumulator in tensor
//      memory; Pi is applied as fp16 hi + lo parts (about 22 bits).
//   3. epilogue (tcgen05.ld, 32 columns): u = sqrt(d) y/||x||; the code comes
//      from a 256-cell table over u in [-8, 8) (one 16-byte shared load: the
//      boundary of the cell, the code below it and both centroids); a u within
//      4e-6 of the boundary is flagged.  Keys: r' = y sqrt(d)/fp16(||x||) -
//      c[code] (the residual in unit-variance units) -> fp16 hi + lo tiles.
//      Flagged codes go through a shared queue; one warp per entry re-decides
//      it from a double-float y and norm and patches the stored word, the
//      residual tiles and the residual norm (rare: about 1e-5 of the codes).
//   4. keys: z = r' S^T as hi*hi + lo*hi + hi*lo fp16 MMAs (about 1e-7 of ||r'||
//      accurate); a |z_p| below 2e-5 ||r'|| is re-decided the same way, one
//      warp per entry: (S Pi)_p x - fp16(||x||)/sqrt(d) * S_p c[code] in
//      double-float.
//   5. the record (codes, signs, fp16 norms) is stored at its page slot.
// Supported here: bf16 or fp32 inputs (fp32 x is split into fp16 hi + lo and
// takes a third MMA set), d = 128, split 64, m multiple of 32 (<= 128), the
// bit-width combinations instantiated below; the rest runs tq_quantize.cu.

#include "tq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

constexpr int kRows = 128;
constexpr int kTmemCols = 256;            // y: columns 0..127, z: 128..255
constexpr float kCodeGuard = 4e-6f;
constexpr float kSignGuard = 2e-5f;
constexpr int kWaitLimit = 1 << 22;
constexpr float kSqrtD = 11.313708498984761f;
constexpr double kSqrtD64 = 11.313708498984760390;
constexpr float kInvSqrtDHi = 0.0883883461356163f;     // fp32(1/sqrt(128))
constexpr float kInvSqrtDLo = 1.512702185735293e-09f;  // 1/sqrt(128) - kInvSqrtDHi

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffPIH = 0;
constexpr int kOffPIL = 32768;
constexpr int kOffSH = 65536;
constexpr int kOffSL = 98304;
constexpr int kOffX = 131072;     // x tile, then the r' low-part tile
constexpr int kOffRH = 163840;    // r' high-part tile

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, fp32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_f16(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}
// Descriptor of k-step s (16 channels) of a 128-channel K-major tile of `rows` rows.
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int s) {
  return sdesc(tile + (s >> 2) * rows * 128 + (s & 3) * 32);
}
// Byte offset of the 16-byte chunk (row, channels 8c..8c+7) in a swizzled tile of `rows` rows.
__device__ __forceinline__ uint32_t swz_chunk(int row, int c, int rows) {
  return (c >> 3) * rows * 128 + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------------------
// double-float helpers
// ---------------------------------------------------------------------------
struct DF {
  float h, l;
};
__device__ __forceinline__ DF two_sum(float a, float b) {
  float s = a + b, bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  DF s = two_sum(a.h, b.h);
  float e = s.l + a.l + b.l;
  float h = s.h + e;
  return {h, e - (h - s.h)};
}
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  float p = a.h * b.h;
  float e = fmaf(a.h, b.h, -p);
  e = fmaf(a.h, b.l, fmaf(a.l, b.h, e));
  float h = p + e;
  return {h, e - (h - p)};
}
__device__ __forceinline__ DF df_fma_acc(DF acc, float ah, float al, float x) {   // acc + (ah + al) * x
  float p = ah * x;
  float e = fmaf(ah, x, -p);
  DF s = two_sum(acc.h, p);
  float l = s.l + acc.l + e + al * x;
  float h = s.h + l;
  return {h, l - (h - s.h)};
}
__device__ __forceinline__ double df_to_d(DF a) { return static_cast<double>(a.h) + static_cast<double>(a.l); }

// fp16 of the double-float value hi + lo >= 0, rounded to nearest even.
__device__ __half df_to_half(float hi, float lo) {
  __half h = __float2half_rn(hi);
  float back = __half2float(h);
  if (back == hi || lo == 0.0f || isinf(back)) return h;
  unsigned short bits = __half_as_ushort(h);
  __half nb = __ushort_as_half(hi > back ? static_cast<unsigned short>(bits + 1) : static_cast<unsigned short>(bits - 1));
  float nbf = __half2float(nb);
  if (hi != 0.5f * (back + nbf)) return h;
  return ((lo > 0.0f) == (nbf > back)) ? nb : h;
}

// ---------------------------------------------------------------------------
// stored code format (see tq.h), for the 32 channels of one quarter of a
// vector: they occupy exactly B consecutive words of the code area
// ---------------------------------------------------------------------------
template <int B>
__device__ __forceinline__ void put_code_q(uint32_t (&w)[4], int c, uint32_t code) {
  if (B == 3) {
    const int o = c >> 3, j = c & 7;
    if (j < 6) {
      const int pos = 24 * o + 4 * j;
      w[pos >> 5] |= code << (pos & 31);
    } else {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int pos = 24 * o + 8 * q + 3 + 4 * (j - 6);
        w[pos >> 5] |= ((code >> q) & 1u) << (pos & 31);
      }
    }
  } else {
    const uint32_t v = (B == 4) ? (code >= 8 ? code - 8 : 15 - code) : code;
    const int pos = B * c;
    w[pos >> 5] |= v << (pos & 31);
  }
}
template <int B>
__device__ __forceinline__ void clear_code_q(uint32_t (&w)[4], int c) {
  if (B == 3) {
    const int o = c >> 3, j = c & 7;
    if (j < 6) {
      const int pos = 24 * o + 4 * j;
      w[pos >> 5] &= ~(7u << (pos & 31));
    } else {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int pos = 24 * o + 8 * q + 3 + 4 * (j - 6);
        w[pos >> 5] &= ~(1u << (pos & 31));
      }
    }
  } else {
    const int pos = B * c;
    w[pos >> 5] &= ~(((1u << B) - 1u) << (pos & 31));
  }
}

// Code of channel c of a quarter from its words (rare paths; any bit width).
__device__ int quarter_code(const uint32_t (&w)[4], int b, int c) {
  auto bitsat = [&](int pos, int n) {     // word by selects: no runtime index into w (kept in registers)
    const int k = pos >> 5;
    const uint32_t x = k == 0 ? w[0] : k == 1 ? w[1] : k == 2 ? w[2] : w[3];
    return static_cast<int>((x >> (pos & 31)) & ((1u << n) - 1u));
  };
  if (b == 3) {
    const int o = c >> 3, j = c & 7;
    if (j < 6) return bitsat(24 * o + 4 * j, 3);
    const int s0 = 24 * o + 3 + 4 * (j - 6);
    return bitsat(s0, 1) | (bitsat(s0 + 8, 1) << 1) | (bitsat(s0 + 16, 1) << 2);
  }
  const int v = bitsat(b * c, b);
  if (b == 4) return (v & 8) ? 7 - (v & 7) : 8 + v;
  return v;
}

// Code of channel j of a stored record (rare paths; any bit width).  Reads go
// to L2: the words may have been patched by atomics of other warps.
__device__ int record_code(const uint32_t* cw, int bh, int bl, int j) {
  const int grp = j < 64 ? 0 : 1, b = grp ? bl : bh, c = grp ? j - 64 : j, base = grp ? 64 * bh : 0;
  auto bitsat = [&](int off, int n) {
    return static_cast<int>((__ldcg(cw + (off >> 5)) >> (off & 31)) & ((1u << n) - 1u));
  };
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

// Replace the code of channel j (old -> nu) in a stored record; fields never
// straddle a word, and XOR patches from several warps commute.
__device__ void patch_code(uint32_t* cw, int bh, int bl, int j, int old, int nu) {
  const int grp = j < 64 ? 0 : 1, b = grp ? bl : bh, c = grp ? j - 64 : j, base = grp ? 64 * bh : 0;
  if (b == 3) {
    const int ob = base + 24 * (c >> 3), i = c & 7;
    const uint32_t dx = static_cast<uint32_t>(old ^ nu);
    if (i < 6) {
      const int pos = ob + 4 * i;
      atomicXor(cw + (pos >> 5), dx << (pos & 31));
    } else {
      for (int k = 0; k < 3; ++k) {
        const int pos = ob + 3 + 4 * (i - 6) + 8 * k;
        if ((dx >> k) & 1u) atomicXor(cw + (pos >> 5), 1u << (pos & 31));
      }
    }
    return;
  }
  auto sv = [&](int code) { return b == 4 ? (code >= 8 ? code - 8 : 15 - code) : code; };
  const int pos = base + b * c;
  atomicXor(cw + (pos >> 5), static_cast<uint32_t>(sv(old) ^ sv(nu)) << (pos & 31));
}

// Sum of a double-float over the warp (every lane gets a sum; lane 0's is used).
__device__ __forceinline__ DF warp_df_sum(DF v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    v = df_add(v, DF{__shfl_xor_sync(0xffffffffu, v.h, off), __shfl_xor_sync(0xffffffffu, v.l, off)});
  return v;
}

// The four channels 4*lane.. of a row (bf16 or fp32 input).
__device__ __forceinline__ void lane_x4(const void* xrow, bool f32, int lane, float (&xv)[4]) {
  if (f32) {
    const float4 r = reinterpret_cast<const float4*>(xrow)[lane];
    xv[0] = r.x, xv[1] = r.y, xv[2] = r.z, xv[3] = r.w;
    return;
  }
  const uint2 r = reinterpret_cast<const uint2*>(xrow)[lane];
  xv[0] = __uint_as_float(r.x << 16);
  xv[1] = __uint_as_float(r.x & 0xFFFF0000u);
  xv[2] = __uint_as_float(r.y << 16);
  xv[3] = __uint_as_float(r.y & 0xFFFF0000u);
}
// x^2 as a double-float (exact).
__device__ __forceinline__ DF df_sq(float x) {
  const float p = x * x;
  return {p, fmaf(x, x, -p)};
}

// Exact code of channel ch (warp-cooperative): y = (Pi_ch hi + lo) . x and
// ||x||^2 in double-float, u = sqrt(d) y/||x|| compared with the fp64
// boundaries.  Lane 0 patches the stored code (the fast path's code `old`,
// stored before a block barrier) when it differs and, for keys,
// the residual tiles and the residual norm partial.
__device__ __noinline__ void refine_code_item(const void* xrow, bool f32, const float* pidf_row, uint32_t* cw, int bh,
                                              int bl, int ch, int old, const double* t64, int nb, const float* cent,
                                              bool key,
                                              float n16f, unsigned char* smem, float* rho2_slot, int row, int lane,
                                              unsigned long long* counter) {
  float xv[4];
  lane_x4(xrow, f32, lane, xv);
  const float4* pr = reinterpret_cast<const float4*>(pidf_row) + 2 * lane;
  const float4 p0 = pr[0], p1 = pr[1];
  DF yd{0.f, 0.f}, n2{0.f, 0.f};
  yd = df_fma_acc(yd, p0.x, p0.y, xv[0]);
  yd = df_fma_acc(yd, p0.z, p0.w, xv[1]);
  yd = df_fma_acc(yd, p1.x, p1.y, xv[2]);
  yd = df_fma_acc(yd, p1.z, p1.w, xv[3]);
#pragma unroll
  for (int k = 0; k < 4; ++k) n2 = df_add(n2, df_sq(xv[k]));
  yd = warp_df_sum(yd);
  n2 = warp_df_sum(n2);
  if (lane != 0) return;
  const double n64 = sqrt(df_to_d(n2));
  const double u64 = n64 > 0.0 ? kSqrtD64 * df_to_d(yd) / n64 : 0.0;
  int code = 0;
  for (int k = 0; k < nb; ++k) code += u64 >= t64[k];
  atomicAdd(counter, 1ULL);
  if (code == old) return;
  patch_code(cw, bh, bl, ch, old, code);
  if (key && n16f > 0.0f) {          // with a zero fp16 norm the residual does not use the code
    const float r = (yd.h + yd.l) * (kSqrtD / n16f) - cent[code];
    const uint32_t off = swz_chunk(row, ch >> 3, kRows) + (ch & 7) * 2;
    __half* ph = reinterpret_cast<__half*>(smem + kOffRH + off);
    __half* pl = reinterpret_cast<__half*>(smem + kOffX + off);
    const float rold = __half2float(*ph) + __half2float(*pl);
    const __half hh = __float2half_rn(r);
    *ph = hh;
    *pl = __float2half_rn(r - __half2float(hh));
    atomicAdd(rho2_slot, r * r - rold * rold);
  }
}

// Exact sign bit of projection p (warp-cooperative):
// (S Pi)_p x - fp16(||x||)/sqrt(d) * S_p c[code] in double-float, with the
// codes read back from the stored record.  Lane 0 patches the stored bit.
__device__ __noinline__ void refine_sign_item(const void* xrow, bool f32, const float* arow, const float* srow,
                                              const uint32_t* cw, int bh, int bl, const float* ch, const float* cl,
                                              float n16f, uint32_t* sw, int bit, int lane,
                                              unsigned long long* counter) {
  float xv[4];
  lane_x4(xrow, f32, lane, xv);
  const float4* ar = reinterpret_cast<const float4*>(arow) + 2 * lane;
  const float4* sr = reinterpret_cast<const float4*>(srow) + 2 * lane;
  const float4 a0 = ar[0], a1 = ar[1], s0 = sr[0], s1 = sr[1];
  const float ah[4] = {a0.x, a0.z, a1.x, a1.z}, al[4] = {a0.y, a0.w, a1.y, a1.w};
  const float sh[4] = {s0.x, s0.z, s1.x, s1.z}, sl[4] = {s0.y, s0.w, s1.y, s1.w};
  DF d1{0.f, 0.f}, d2{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * lane + k;
    const int cj = record_code(cw, bh, bl, j) + (j < 64 ? 0 : 16);
    d1 = df_fma_acc(d1, ah[k], al[k], xv[k]);
    d2 = df_add(d2, df_mul(DF{sh[k], sl[k]}, DF{ch[cj], cl[cj]}));
  }
  d1 = warp_df_sum(d1);
  d2 = warp_df_sum(d2);
  if (lane != 0) return;
  const DF f = df_mul(DF{n16f, 0.f}, DF{kInvSqrtDHi, kInvSqrtDLo});
  const DF fz = df_mul(f, d2);
  const DF z = df_add(d1, DF{-fz.h, -fz.l});
  const uint32_t nb = (z.h > 0.0f || (z.h == 0.0f && z.l >= 0.0f)) ? 1u : 0u;
  atomicAdd(counter, 1ULL);
  if (((__ldcg(sw) >> bit) & 1u) != nb) atomicXor(sw, 1u << bit);
}

// Code-assignment cells: per channel group 256 cells of width 1/16 over
// u in [-8, 8).  A cell keeps the one boundary t that matters for u inside it
// (the boundary in the cell, else the nearest), the code for u < t and the
// centroids for u < t and u >= t; boundaries are >= 0.25 apart for b <= 4.
struct Cell {
  float t;
  int code;
  float c_below;
  float c_above;
};
constexpr int kCells = 256;
constexpr int kThreadsTC4 = 512;

__device__ void build_cells(Cell* cells, const GroupBook& gb, int idx) {
  const float lo = -8.0f + idx * (1.0f / 16.0f), hi = lo + 1.0f / 16.0f;
  int inside = -1, nearest = 0, below = 0;
  float best = INFINITY;
  for (int k = 0; k < gb.nb; ++k) {
    const float t = gb.t[k];
    if (t < lo) ++below;
    if (t >= lo && t < hi) inside = k;
    const float dist = t < lo ? lo - t : (t >= hi ? t - hi : 0.0f);
    if (dist < best) { best = dist; nearest = k; }
  }
  Cell c;
  if (inside >= 0) {
    c.t = gb.t[inside];
    c.code = inside;                       // boundaries below t_inside: exactly `inside` of them
  } else {
    c.t = gb.t[nearest];
    c.code = c.t < lo ? below - 1 : below; // u >= t always (t below) or never (t above)
  }
  c.c_below = gb.c[max(c.code, 0)];
  c.c_above = gb.c[min(c.code + 1, 15)];
  cells[idx] = c;
}

// shared memory beyond the tiles
constexpr int kOffCells = 196608;                 // 4 groups x 256 cells x 16 B
constexpr int kOffMisc4 = kOffCells + 4 * kCells * 16;

// Epilogue of one quarter (32 channels of group width B) of one row: codes,
// the smallest |u - t| (the caller builds the near-boundary mask when it is
// under the guard, rarely) and, for keys, the residual as fp16 hi + lo pairs.
template <int B, bool KEY>
__device__ __forceinline__ void quarter_epilogue(const float (&v)[32], const Cell* cells, float ku, float kr,
                                                 float sub, uint32_t (&words)[4], float& dmin, float& rho2,
                                                 uint32_t (&rh)[16], uint32_t (&rl)[16]) {
  float r_even = 0.0f;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float u = v[c] * ku;
    const int g = min(max(__float2int_rd(fmaf(u, 16.0f, 128.0f)), 0), kCells - 1);
    const float4 cell = reinterpret_cast<const float4*>(cells)[g];
    const bool ge = u >= cell.x;
    const int code = __float_as_int(cell.y) + (ge ? 1 : 0);
    dmin = fminf(dmin, fabsf(u - cell.x));
    put_code_q<B>(words, c, static_cast<uint32_t>(code));
    if (KEY) {
      const float r = fmaf(v[c], kr, -sub * (ge ? cell.w : cell.z));
      rho2 = fmaf(r, r, rho2);
      if (c & 1) {
        const __half2 h = __floats2half2_rn(r_even, r);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(r_even - hf.x, r - hf.y);
        rh[c >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        rl[c >> 1] = *reinterpret_cast<const uint32_t*>(&l);
      } else {
        r_even = r;
      }
    }
  }
}

// Misc shared area (after the cells).
constexpr int kQueueCap = 128;
constexpr int kMiscQn = 20, kMiscT64 = 64, kMiscCent = 576, kMiscCentLo = 832, kMiscRedSH = 1152,
              kMiscRedSL = 3200, kMiscRedM = 5248, kMiscRedR = 7296, kMiscN16 = 9344, kMiscCodePtr = 9856,
              kMiscSignPtr = 10880, kMiscQueue = 11904, kMiscBytes = 12544;
constexpr int kSmemBytes4 = kOffMisc4 + kMiscBytes + 1024;   // + alignment slack
static_assert(kSmemBytes4 <= 232448, "shared memory per block");

// ---------------------------------------------------------------------------
// the kernel: 16 warps; warp w reads tensor-memory lanes 32*(w%4).. (rows) and
// handles channel quarter w/4 of those rows
// ---------------------------------------------------------------------------
template <int KBH, int KBL, int VBH, int VBL>
__global__ void __launch_bounds__(kThreadsTC4, 1) quantize_tc_kernel(QuantizeArgs ka, QuantizeArgs va, int nk_tiles,
                                                                     int nv_tiles) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // aligned by an offset on the shared array itself, so that every access
  // through smem stays a shared-memory access (not a generic one)
  unsigned char* smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Cell* cells = reinterpret_cast<Cell*>(smem + kOffCells);
  unsigned char* misc = smem + kOffMisc4;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(misc);   // [0] tables, [1] mma
  unsigned long long* xbar = reinterpret_cast<unsigned long long*>(misc + 24);   // x prefetch
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 16);
  int* qn = reinterpret_cast<int*>(misc + kMiscQn);
  double* t64s = reinterpret_cast<double*>(misc + kMiscT64);                  // [4][16]
  float* cents = reinterpret_cast<float*>(misc + kMiscCent);                  // [4][16]
  float* centl = reinterpret_cast<float*>(misc + kMiscCentLo);                // [4][16]
  float* rownf = reinterpret_cast<float*>(misc + kMiscRedSH);                 // [128] fp32 norm
  float* rowscale = reinterpret_cast<float*>(misc + kMiscRedSL);              // [128] power-of-two x scale
  unsigned short** rnormptr = reinterpret_cast<unsigned short**>(misc + kMiscRedM);   // [128] rnorm slot or null
  unsigned short** normptr = rnormptr + kRows;                                       // [128] norm slot or null
  float* red_r = reinterpret_cast<float*>(misc + kMiscRedR);
  float* rown16 = reinterpret_cast<float*>(misc + kMiscN16);                  // [128]
  uint32_t** codeptr = reinterpret_cast<uint32_t**>(misc + kMiscCodePtr);     // [128], null: no record
  uint32_t** signptr = reinterpret_cast<uint32_t**>(misc + kMiscSignPtr);     // [128]
  uint32_t* queue = reinterpret_cast<uint32_t*>(misc + kMiscQueue);           // [kQueueCap]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp >> 2;
  const int row = 32 * (warp & 3) + lane;
  const int m = ka.m;
  const bool have_k = nk_tiles > 0;

  for (int i = tid; i < 4 * kCells; i += kThreadsTC4) {
    const int grp = i / kCells;
    const KindLayout& L = grp < 2 ? ka.lay : va.lay;
    build_cells(cells + grp * kCells, L.g[grp & 1], i % kCells);
  }
  if (tid < 64) {
    const int grp = tid >> 4, k = tid & 15;
    const GroupBook& gb = (grp < 2 ? ka.lay : va.lay).g[grp & 1];
    t64s[tid] = gb.t64[k];
    cents[tid] = gb.c[k];
    centl[tid] = gb.c_lo[k];
  }
  if (tid == 0) *qn = 0;
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init(smem_u32(xbar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t bytes = 2 * 32768 + (have_k ? 2 * m * 256 : 0);
    mbar_arrive_tx(smem_u32(&bars[0]), bytes);
    bulk_g2s(sbase + kOffPIH, ka.tab.pih_sw, 32768, smem_u32(&bars[0]));
    bulk_g2s(sbase + kOffPIL, ka.tab.pil_sw, 32768, smem_u32(&bars[0]));
    if (have_k) {
      bulk_g2s(sbase + kOffSH, ka.tab.sh_sw, m * 256, smem_u32(&bars[0]));
      bulk_g2s(sbase + kOffSL, ka.tab.sl_sw, m * 256, smem_u32(&bars[0]));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // a wait that gives up sets the flag in every thread (uniform exit)
  bool failed = __syncthreads_or(!mbar_wait(smem_u32(&bars[0]), 0)) != 0;
  uint32_t phase = 0, xphase = 0;
  const uint32_t trow = tmem + ((32u * (warp & 3)) << 16);

  const int ntiles = nk_tiles + nv_tiles;
  // bf16 tiles are contiguous (128 rows x 256 B): the next one is bulk-copied
  // into the residual tile once that is free, so a tile starts from shared
  // memory.  Returns whether a copy was issued (same answer in every thread).
  auto prefetch_x = [&](int nt) {
    if (nt >= ntiles) return false;
    const QuantizeArgs& an = nt < nk_tiles ? ka : va;
    if (an.f32) return false;
    const long long nvec_n = static_cast<long long>(an.batch) * an.n_new * an.H;
    const long long g0 = static_cast<long long>(nt < nk_tiles ? nt : nt - nk_tiles) * kRows;
    const uint32_t rows = static_cast<uint32_t>(nvec_n - g0 < kRows ? nvec_n - g0 : kRows);
    if (tid == 0) {
      mbar_arrive_tx(smem_u32(xbar), rows * kD * 2);
      bulk_g2s(sbase + kOffRH, static_cast<const unsigned char*>(an.x) + g0 * kD * 2, rows * kD * 2, smem_u32(xbar));
    }
    return true;
  };
  bool xpref = !failed && prefetch_x(blockIdx.x);
  for (int tile = blockIdx.x; tile < ntiles && !failed; tile += gridDim.x) {
    const bool key = tile < nk_tiles;
    const QuantizeArgs& a = key ? ka : va;
    const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
    const long long gv0 = static_cast<long long>(key ? tile : tile - nk_tiles) * kRows;
    const bool valid = gv0 + row < nvec;
    const bool f32 = a.f32 != 0;
    const bool sk = key && a.lay.qjl;              // keys with residual signs
    const size_t esz = f32 ? 4 : 2;
    const unsigned char* xbase = static_cast<const unsigned char*>(a.x) + static_cast<size_t>(gv0) * kD * esz;
    auto xrow_of = [&](int r) { return static_cast<const void*>(xbase + static_cast<size_t>(r) * kD * esz); };

    // ---- 1. rows -> statistics -> scaled fp16 tile (16 lanes per row) ------
    const bool xsm = xpref;                  // this tile's x is in the residual tile
    if (xsm) {
      if (__syncthreads_or(!mbar_wait(smem_u32(xbar), xphase))) {
        failed = true;
        if (tid == 0) atomicOr(a.tab.err, kErrTimeout);
      }
      xphase ^= 1;
      xpref = false;
    }
#pragma unroll 1
    for (int pass = 0; pass < kRows / 32; ++pass) {
      const int r = 32 * pass + 2 * warp + (lane >> 4), c = lane & 15;   // row, channels 8c..8c+7
      const bool rv = gv0 + r < nvec;
      float xv[8];
      if (f32) {
        const float4* src = reinterpret_cast<const float4*>(xbase + static_cast<size_t>(r) * kD * 4) + 2 * c;
        const float4 u0 = rv ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 u1 = rv ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        xv[0] = u0.x, xv[1] = u0.y, xv[2] = u0.z, xv[3] = u0.w, xv[4] = u1.x, xv[5] = u1.y, xv[6] = u1.z, xv[7] = u1.w;
      } else {
        uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
        if (rv)
          w4 = xsm ? *reinterpret_cast<const uint4*>(smem + kOffRH + r * kD * 2 + 16 * c)
                   : *reinterpret_cast<const uint4*>(xbase + static_cast<size_t>(r) * kD * 2 + 16 * c);
        const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xv[2 * k] = __uint_as_float(ww[k] << 16);
          xv[2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
        }
      }
      float s0 = 0.f, s1 = 0.f, mx = 0.f;
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        s0 = fmaf(xv[k], xv[k], s0);
        s1 = fmaf(xv[k + 1], xv[k + 1], s1);
        mx = fmaxf(mx, fmaxf(fabsf(xv[k]), fabsf(xv[k + 1])));
      }
      float ss = s0 + s1;
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {      // the row's 16 lanes
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      // fp32 norm (relative error < 4e-6); the fp16 norm must round the exact
      // value, so a norm within 1e-5 of an fp16 midpoint is recomputed from a
      // double-float sum of the exact squares
      float nf = ss > 0.0f ? sqrtf(ss) : 0.0f;
      __half h = __float2half_rn(nf);
      bool near_mid = false;
      if (nf > 0.0f) {
        const float hb = __half2float(h);
        const unsigned short hbits = __half_as_ushort(h);
        const float up = __half2float(__ushort_as_half(static_cast<unsigned short>(hbits + 1)));
        const float dn = hbits ? __half2float(__ushort_as_half(static_cast<unsigned short>(hbits - 1))) : 0.0f;
        const float tol = 1e-5f * nf;
        near_mid = fabsf(nf - 0.5f * (hb + up)) < tol || fabsf(nf - 0.5f * (hb + dn)) < tol;
      }
      if (__any_sync(0xffffffffu, near_mid)) {
        DF n2{0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 8; ++k) n2 = df_add(n2, df_sq(xv[k]));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1)
          n2 = df_add(n2, DF{__shfl_xor_sync(0xffffffffu, n2.h, off), __shfl_xor_sync(0xffffffffu, n2.l, off)});
        if (near_mid) {
          const float rr = sqrtf(n2.h);
          const float rl = (fmaf(-rr, rr, n2.h) + n2.l) / (2.0f * rr);
          nf = rr + rl;
          h = df_to_half(nf, rl - (nf - rr));
        }
      }
      float xs = 1.0f;
      if (mx > 0.0f) {
        int e;
        frexpf(mx, &e);
        xs = ldexpf(1.0f, 14 - e);
      }
      // fp16 x * 2^k (exact for bf16); fp32 input also gets the remainder as a
      // second fp16 tile (in the residual tile, free until the epilogue)
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = xv[2 * k] * xs, x1 = xv[2 * k + 1] * xs;
        const __half2 ph = __floats2half2_rn(x0, x1);
        hv[k] = *reinterpret_cast<const uint32_t*>(&ph);
        if (f32) {
          const __half2 pl = __floats2half2_rn(x0 - __low2float(ph), x1 - __high2float(ph));
          lv[k] = *reinterpret_cast<const uint32_t*>(&pl);
        }
      }
      const uint32_t off = swz_chunk(r, c, kRows);
      *reinterpret_cast<uint4*>(smem + kOffX + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      if (f32) *reinterpret_cast<uint4*>(smem + kOffRH + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      if (c == 0) {
        rownf[r] = nf;
        rown16[r] = __half2float(h);
        rowscale[r] = xs;
      }
    }
    // record location of every row: one thread per row
    if (tid < kRows) {
      const int r = tid;
      unsigned char* rec = nullptr;
      int slot = 0;
      if (gv0 + r < nvec) {
        int hh, t, b;
        const long long gv = gv0 + r;
        if (nvec < (1LL << 31)) {          // 32-bit division when it fits
          const uint32_t g32 = static_cast<uint32_t>(gv), H32 = static_cast<uint32_t>(a.H);
          const uint32_t bt = g32 / H32;
          hh = static_cast<int>(g32 - bt * H32);
          b = static_cast<int>(bt / static_cast<uint32_t>(a.n_new));
          t = static_cast<int>(bt - static_cast<uint32_t>(b) * static_cast<uint32_t>(a.n_new));
        } else {
          const long long bt = gv / a.H;
          hh = static_cast<int>(gv % a.H);
          t = static_cast<int>(bt % a.n_new);
          b = static_cast<int>(bt / a.n_new);
        }
        const int pos = a.start_pos[b] + t;
        const int blk = pos >> 4;
        if (pos < 0 || blk >= a.maxp) {
          atomicOr(a.tab.err, kErrBlock);
        } else {
          const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.tab.err, kErrPage);
          } else {
            rec = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(hh) * a.lay.block_bytes;
            slot = pos & 15;
          }
        }
      }
      codeptr[r] = rec ? reinterpret_cast<uint32_t*>(rec + slot * a.lay.code_bytes) : nullptr;
      signptr[r] = rec ? reinterpret_cast<uint32_t*>(rec + a.lay.off_signs + slot * (m / 8)) : nullptr;
      rnormptr[r] = (rec && sk) ? reinterpret_cast<unsigned short*>(rec + a.lay.off_rnorm) + slot : nullptr;
      normptr[r] = rec ? reinterpret_cast<unsigned short*>(rec + a.lay.off_norm) + slot : nullptr;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- 2. y = x Pi^T ------------------------------------------------------
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma_f16(tmem, kdesc(sbase + kOffX, kRows, s), kdesc(sbase + kOffPIH, kRows, s), idesc_f16(128), s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma_f16(tmem, kdesc(sbase + kOffX, kRows, s), kdesc(sbase + kOffPIL, kRows, s), idesc_f16(128), 1u);
      if (f32) {
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_f16(tmem, kdesc(sbase + kOffRH, kRows, s), kdesc(sbase + kOffPIH, kRows, s), idesc_f16(128), 1u);
      }
      umma_commit(smem_u32(&bars[1]));
    }
    if (__syncthreads_or(!mbar_wait(smem_u32(&bars[1]), phase))) {
      failed = true;
      if (tid == 0) atomicOr(a.tab.err, kErrTimeout);
    }
    phase ^= 1;
    tc_fence_after();
    // the residual tile is free now unless this tile still needs it for r'
    if (!sk) xpref = prefetch_x(tile + gridDim.x);
    const float nf = rownf[row], n16f = rown16[row], xs_scale = rowscale[row];
    if (q == 0 && normptr[row]) *normptr[row] = __half_as_ushort(__float2half_rn(n16f));   // exact: n16f is fp16

    // ---- 3. codes and residual of this quarter -------------------------------
    const int grp = q < 2 ? 0 : 1;
    const int gslot = (key ? 0 : 2) + grp;
    const int bh = key ? KBH : VBH, bl = key ? KBL : VBL;
    uint32_t* const cp = codeptr[row];
    uint32_t near = 0;
    float dmin = INFINITY;
    uint32_t words[4] = {0u, 0u, 0u, 0u};   // this quarter's codes as stored
    {
      const float inv = 1.0f / (xs_scale * kPiScale);
      const float ku = nf > 0.0f ? inv * (kSqrtD / nf) : 0.0f;
      // a zero fp16 norm leaves the residual equal to y (any positive scale
      // gives the same signs), so it is formed without the centroids
      const float kr = n16f > 0.0f ? inv * (kSqrtD / n16f) : ku;
      const float sub = n16f > 0.0f ? 1.0f : 0.0f;
      uint32_t rh[16], rl[16];
      float rho2 = 0.0f;
      float v[32];
      tmem_ld32(trow + 32 * q, v);
      const Cell* cg = cells + gslot * kCells;
      if (sk) {
        if (grp == 0) quarter_epilogue<KBH, true>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
        else quarter_epilogue<KBL, true>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
      } else if (key) {
        if (grp == 0) quarter_epilogue<KBH, false>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
        else quarter_epilogue<KBL, false>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
      } else {
        if (grp == 0) quarter_epilogue<VBH, false>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
        else quarter_epilogue<VBL, false>(v, cg, ku, kr, sub, words, dmin, rho2, rh, rl);
      }
      // near-boundary mask from the tensor-memory values again (warp-uniform:
      // the load is collective; a row whose dmin passed gets no bits)
      if (__any_sync(0xffffffffu, dmin < kCodeGuard)) {
        float w2[32];
        tmem_ld32(trow + 32 * q, w2);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float u = w2[c] * ku;
          const int g = min(max(__float2int_rd(fmaf(u, 16.0f, 128.0f)), 0), kCells - 1);
          near |= (fabsf(u - cg[g].t) < kCodeGuard ? 1u : 0u) << c;
        }
      }
      if (!valid || nf == 0.0f || !cp) near = 0;
      if (sk) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = swz_chunk(row, 4 * q + c, kRows);
          *reinterpret_cast<uint4*>(smem + kOffRH + off) = make_uint4(rh[4 * c], rh[4 * c + 1], rh[4 * c + 2], rh[4 * c + 3]);
          *reinterpret_cast<uint4*>(smem + kOffX + off) = make_uint4(rl[4 * c], rl[4 * c + 1], rl[4 * c + 2], rl[4 * c + 3]);
        }
        red_r[q * 128 + row] = rho2;
      }
      if (cp) {
        const int woff = q < 2 ? q * bh : 2 * bh + (q - 2) * bl;
        const int nw = grp ? bl : bh;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (w < nw) cp[woff + w] = words[w];
      }
    }

    // ---- 3b. exact re-decision of flagged codes (rare; whole CTA) -----------
    // (the block barrier orders the stored words before the patches: no fence)
    if (__syncthreads_or(near != 0)) {
      uint32_t mine = near;
      for (;;) {
        while (mine) {
          const int idx = atomicAdd(qn, 1);
          if (idx >= kQueueCap) break;
          const int c = __ffs(mine) - 1;
          mine &= mine - 1;
          const uint32_t old = static_cast<uint32_t>(quarter_code(words, grp ? bl : bh, c));
          queue[idx] = static_cast<uint32_t>(row) | (static_cast<uint32_t>(32 * q + c) << 8) | (old << 16);
        }
        __syncthreads();
        const int n = min(*qn, kQueueCap);
        for (int i = warp; i < n; i += kThreadsTC4 / 32) {
          const int r = static_cast<int>(queue[i] & 255u), ch = static_cast<int>((queue[i] >> 8) & 255u);
          const int old = static_cast<int>(queue[i] >> 16);
          const int gs = (key ? 0 : 2) + (ch < 64 ? 0 : 1);
          const int b = ch < 64 ? bh : bl;
          refine_code_item(xrow_of(r), f32, a.tab.pi_df + ch * kD * 2, codeptr[r], bh, bl, ch, old,
                           t64s + gs * 16, (1 << b) - 1, cents + gs * 16, sk, rown16[r], smem, &red_r[r], r, lane,
                           &a.tab.counters[0]);
        }
        __syncthreads();
        if (tid == 0) *qn = 0;
        if (!__syncthreads_or(mine != 0)) break;
      }
    }

    // ---- 4. keys: z = r' S^T and the sign bits -------------------------------
    if (sk) {
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t zt = tmem + 128;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_f16(zt, kdesc(sbase + kOffRH, kRows, s), kdesc(sbase + kOffSH, m, s), idesc_f16(m), s > 0);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_f16(zt, kdesc(sbase + kOffX, kRows, s), kdesc(sbase + kOffSH, m, s), idesc_f16(m), 1u);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          umma_f16(zt, kdesc(sbase + kOffRH, kRows, s), kdesc(sbase + kOffSL, m, s), idesc_f16(m), 1u);
        umma_commit(smem_u32(&bars[1]));
      }
      if (__syncthreads_or(!mbar_wait(smem_u32(&bars[1]), phase))) {
        failed = true;
        if (tid == 0) atomicOr(a.tab.err, kErrTimeout);
      }
      phase ^= 1;
      tc_fence_after();
      xpref = prefetch_x(tile + gridDim.x);      // the z MMA has read the residual tile
      const float rho = sqrtf((red_r[row] + red_r[128 + row]) + (red_r[256 + row] + red_r[384 + row]));
      uint32_t nearz = 0;
      if (32 * q < m) {
        float v[32];
        tmem_ld32(trow + 128 + 32 * q, v);
        const float guard = kSignGuard * rho;
        uint32_t word = 0;
        float amin = INFINITY;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          word |= ((~__float_as_uint(v[k])) >> 31) << k;
          amin = fminf(amin, fabsf(v[k]));
        }
        if (__any_sync(0xffffffffu, amin < guard)) {     // rare: the near-zero mask
#pragma unroll
          for (int k = 0; k < 32; ++k) nearz |= (fabsf(v[k]) < guard ? 1u : 0u) << k;
        }
        uint32_t* const sp = signptr[row];
        if (!sp) nearz = 0;
        if (sp) sp[q] = word;
      }
      if (__syncthreads_or(nearz != 0)) {
        uint32_t mine = nearz;
        for (;;) {
          while (mine) {
            const int idx = atomicAdd(qn, 1);
            if (idx >= kQueueCap) break;
            const int k = __ffs(mine) - 1;
            mine &= mine - 1;
            queue[idx] = static_cast<uint32_t>(row) | (static_cast<uint32_t>(32 * q + k) << 8);
          }
          __syncthreads();
          const int n = min(*qn, kQueueCap);
          for (int i = warp; i < n; i += kThreadsTC4 / 32) {
            const int r = static_cast<int>(queue[i] & 255u), p = static_cast<int>(queue[i] >> 8);
            refine_sign_item(xrow_of(r), f32, a.tab.a_df + static_cast<long long>(p) * kD * 2,
                             a.tab.s_df + static_cast<long long>(p) * kD * 2, codeptr[r], KBH, KBL, cents, centl,
                             rown16[r], signptr[r] + (p >> 5), p & 31, lane, &a.tab.counters[1]);
          }
          __syncthreads();
          if (tid == 0) *qn = 0;
          if (!__syncthreads_or(mine != 0)) break;
        }
      }
      if (q == 0 && rnormptr[row]) *rnormptr[row] = __half_as_ushort(__float2half_rn(rho * n16f * kInvSqrtDHi));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // a prefetch issued for a tile this CTA no longer runs (after a failure)
  // lands before the CTA can exit (bounded wait)
  if (xpref) (void)mbar_wait(smem_u32(xbar), xphase);
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int KBH, int KBL, int VBH, int VBL>
cudaError_t launch_tc(const QuantizeArgs& k, const QuantizeArgs& v, int nk, int nv, cudaStream_t s) {
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = smem_attr_once(quantize_tc_kernel<KBH, KBL, VBH, VBL>, kSmemBytes4, configured);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = nk + nv;
  const int cap = k.max_ctas > 0 && k.max_ctas < sms ? k.max_ctas : sms;
  const int grid = tiles < cap ? tiles : cap;
  quantize_tc_kernel<KBH, KBL, VBH, VBL><<<grid, kThreadsTC4, kSmemBytes4, s>>>(k, v, nk, nv);
  return cudaGetLastError();
}

}  // namespace

bool launch_quantize_tc(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err) {
  if ((k.x && (k.lay.split != 64 || k.m % 32 || k.m < 32 || k.m > 128)) || (v.x && v.lay.split != 64)) return false;
  if ((reinterpret_cast<uintptr_t>(k.x) | reinterpret_cast<uintptr_t>(v.x)) & 15) return false;
  const long long nk_vec = k.x ? static_cast<long long>(k.batch) * k.n_new * k.H : 0;
  const long long nv_vec = v.x ? static_cast<long long>(v.batch) * v.n_new * v.H : 0;
  if ((nk_vec + kRows - 1) / kRows + (nv_vec + kRows - 1) / kRows > (1LL << 31) - 1) return false;
  const int nk = static_cast<int>((nk_vec + kRows - 1) / kRows);
  const int nv = static_cast<int>((nv_vec + kRows - 1) / kRows);
  // bit widths of the two kinds (a missing kind takes the other's, it has no tiles)
  const KindLayout& kl = k.x ? k.lay : v.lay;
  const KindLayout& vl = v.x ? v.lay : k.lay;
  const int code = kl.g[0].bits * 1000 + kl.g[1].bits * 100 + vl.g[0].bits * 10 + vl.g[1].bits;
  QuantizeArgs kk = k.x ? k : v, vv = v.x ? v : k;
  switch (code) {
    case 3333: *err = launch_tc<3, 3, 3, 3>(kk, vv, nk, nv, s); return true;
    case 4343: *err = launch_tc<4, 3, 4, 3>(kk, vv, nk, nv, s); return true;
    case 3232: *err = launch_tc<3, 2, 3, 2>(kk, vv, nk, nv, s); return true;
    case 4444: *err = launch_tc<4, 4, 4, 4>(kk, vv, nk, nv, s); return true;
    case 2222: *err = launch_tc<2, 2, 2, 2>(kk, vv, nk, nv, s); return true;
    case 4422: *err = launch_tc<4, 4, 2, 2>(kk, vv, nk, nv, s); return true;
    default: return false;
  }
}

}  // namespace tq
