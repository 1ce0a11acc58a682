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
//   1. x quarter -> partial sum of squares and max (reduced over the four
//      threads in shared memory) -> fp32 norm, fp16 norm (exact: values near
//      an fp16 rounding midpoint are recomputed in double-float), fp16 x scaled
//      by a power of two (exact for bf16) in a 128-byte-swizzled K-major tile.
//   2. y = x Pi^T: tcgen05.mma kind::f16, M=128 N=128, accumulator in tensor
//      memory; Pi is applied as fp16 hi + lo parts (about 22 bits).
//   3. epilogue (tcgen05.ld, 32 columns): u = sqrt(d) y/||x||; the code comes
//      from a 256-cell table over u in [-8, 8) (one 16-byte shared load: the
//      boundary of the cell, the code below it and both centroids); a u within
//      4e-6 of the boundary is flagged and re-decided after the unrolled pass
//      from a double-float y and norm.  Keys: r' = y sqrt(d)/fp16(||x||) -
//      c[code] (the residual in unit-variance units) -> fp16 hi + lo tiles.
//   4. keys: z = r' S^T as hi*hi + lo*hi + hi*lo fp16 MMAs (about 1e-7 of ||r'||
//      accurate); a |z_p| below 2e-5 ||r'|| is re-decided exactly as
//      (S Pi)_p x - fp16(||x||)/sqrt(d) * S_p c[code] in double-float.
//   5. the record (codes, signs, fp16 norms) is stored at its page slot.
// Supported here: bf16 inputs, d = 128, split 64, m multiple of 32 (<= 128),
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
constexpr uint32_t kErrTimeout = 8u;
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

// Code of channel j of a stored record (rare paths; any bit width).
__device__ int record_code(const uint32_t* cw, int bh, int bl, int j) {
  const int grp = j < 64 ? 0 : 1, b = grp ? bl : bh, c = grp ? j - 64 : j, base = grp ? 64 * bh : 0;
  auto bitsat = [&](int off, int n) {
    const unsigned long long pair = (static_cast<unsigned long long>(cw[(off >> 5) + 1]) << 32) | cw[off >> 5];
    return static_cast<int>((pair >> (off & 31)) & ((1u << n) - 1u));
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

// Exact code of channel i: y_i = (Pi_i hi + lo) . x and ||x|| in double-float,
// u = sqrt(d) y_i / ||x|| compared with the fp64 boundaries.
__device__ __noinline__ int refine_code(const __nv_bfloat16* x, const float* prow, const double* t64, int nb) {
  DF yd{0.f, 0.f}, n2{0.f, 0.f};
  for (int k = 0; k < kD; ++k) {
    const float xv = __bfloat162float(x[k]);
    yd = df_fma_acc(yd, prow[2 * k], prow[2 * k + 1], xv);
    n2 = df_add(n2, DF{xv * xv, 0.f});        // squares of bf16 values are exact in fp32
  }
  const double n64 = sqrt(df_to_d(n2));
  const double u64 = n64 > 0.0 ? kSqrtD64 * df_to_d(yd) / n64 : 0.0;
  int code = 0;
  for (int k = 0; k < nb; ++k) code += u64 >= t64[k];
  return code;
}

// Exact sign bit of projection p: (S Pi)_p x - fp16(||x||)/sqrt(d) * S_p c[code],
// with the centroid of every channel given as double-float pairs in cdf.
__device__ __noinline__ uint32_t refine_sign(const __nv_bfloat16* x, const float* arow, const float* srow,
                                             const float* cdf, float n16f) {
  DF d1{0.f, 0.f}, d2{0.f, 0.f};
  for (int j = 0; j < kD; ++j) {
    d1 = df_fma_acc(d1, arow[2 * j], arow[2 * j + 1], __bfloat162float(x[j]));
    d2 = df_add(d2, df_mul(DF{srow[2 * j], srow[2 * j + 1]}, DF{cdf[2 * j], cdf[2 * j + 1]}));
  }
  const DF f = df_mul(DF{n16f, 0.f}, DF{kInvSqrtDHi, kInvSqrtDLo});
  const DF fz = df_mul(f, d2);
  const DF z = df_add(d1, DF{-fz.h, -fz.l});
  return (z.h > 0.0f || (z.h == 0.0f && z.l >= 0.0f)) ? 1u : 0u;
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
constexpr int kSmemBytes4 = kOffMisc4 + 8192 + 1024;

// Epilogue of one quarter (32 channels of group width B) of one row.
template <int B, bool KEY>
__device__ __forceinline__ void quarter_epilogue(const float (&v)[32], const Cell* cells, float ku, float kr,
                                                 uint32_t (&words)[4], uint32_t& near, float& rho2,
                                                 uint32_t (&rh)[16], uint32_t (&rl)[16]) {
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float u = v[c] * ku;
    const int g = min(max(__float2int_rd(fmaf(u, 16.0f, 128.0f)), 0), kCells - 1);
    const float4 cell = reinterpret_cast<const float4*>(cells)[g];
    const bool ge = u >= cell.x;
    const int code = __float_as_int(cell.y) + (ge ? 1 : 0);
    near |= (fabsf(u - cell.x) < kCodeGuard ? 1u : 0u) << c;
    put_code_q<B>(words, c, static_cast<uint32_t>(code));
    if (KEY) {
      const float r = fmaf(v[c], kr, -(ge ? cell.w : cell.z));
      rho2 = fmaf(r, r, rho2);
      const __half hh = __float2half_rn(r);
      const __half hl = __float2half_rn(r - __half2float(hh));
      const uint32_t sh = (c & 1) ? 16u : 0u;
      if (!(c & 1)) {
        rh[c >> 1] = 0u;
        rl[c >> 1] = 0u;
      }
      rh[c >> 1] |= static_cast<uint32_t>(__half_as_ushort(hh)) << sh;
      rl[c >> 1] |= static_cast<uint32_t>(__half_as_ushort(hl)) << sh;
    }
  }
}

// Re-decide flagged codes of a quarter exactly and patch words / residual.
template <int B, bool KEY>
__device__ __noinline__ void quarter_refine(const float (&v)[32], uint32_t near, const __nv_bfloat16* xrow,
                                            const float* pi_df, int ch0, const double* t64, int nb, const float* cent,
                                            float kr, uint32_t (&words)[4], float& rho2, uint32_t (&rh)[16],
                                            uint32_t (&rl)[16], unsigned long long* counter) {
  while (near) {
    const int c = __ffs(near) - 1;
    near &= near - 1;
    const int code = refine_code(xrow, pi_df + (ch0 + c) * kD * 2, t64, nb);
    atomicAdd(counter, 1ULL);
#pragma unroll
    for (int c2 = 0; c2 < 32; ++c2) {
      if (c2 != c) continue;
      clear_code_q<B>(words, c2);
      put_code_q<B>(words, c2, static_cast<uint32_t>(code));
      if (KEY) {
        const uint32_t sh = (c2 & 1) ? 16u : 0u;
        const float rold = __half2float(__ushort_as_half(static_cast<unsigned short>(rh[c2 >> 1] >> sh))) +
                           __half2float(__ushort_as_half(static_cast<unsigned short>(rl[c2 >> 1] >> sh)));
        const float r = fmaf(v[c2], kr, -cent[code]);
        rho2 += r * r - rold * rold;
        const __half hh = __float2half_rn(r);
        const __half hl = __float2half_rn(r - __half2float(hh));
        rh[c2 >> 1] = (rh[c2 >> 1] & ~(0xFFFFu << sh)) | (static_cast<uint32_t>(__half_as_ushort(hh)) << sh);
        rl[c2 >> 1] = (rl[c2 >> 1] & ~(0xFFFFu << sh)) | (static_cast<uint32_t>(__half_as_ushort(hl)) << sh);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel: 16 warps; warp w reads tensor-memory lanes 32*(w%4).. (rows) and
// handles channel quarter w/4 of those rows
// ---------------------------------------------------------------------------
template <int KBH, int KBL, int VBH, int VBL>
__global__ void __launch_bounds__(kThreadsTC4, 1) quantize_tc_kernel(QuantizeArgs ka, QuantizeArgs va, int nk_tiles,
                                                                     int nv_tiles) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Cell* cells = reinterpret_cast<Cell*>(smem + kOffCells);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem + kOffMisc4);   // [0] tables, [1] mma
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc4 + 16);
  double* t64s = reinterpret_cast<double*>(smem + kOffMisc4 + 64);                      // [4][16]
  float* cents = reinterpret_cast<float*>(smem + kOffMisc4 + 64 + 512);                 // [4][16]
  float* red_s = reinterpret_cast<float*>(smem + kOffMisc4 + 1024);                     // [4][128]
  float* red_m = red_s + 512;
  float* red_r = red_m + 512;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sp = warp & 3, q = warp >> 2;
  const int row = 32 * sp + lane;
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
    cents[grp * 16 + k] = gb.c[k];
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
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
  bool failed = !mbar_wait(smem_u32(&bars[0]), 0);
  uint32_t phase = 0;
  const uint32_t trow = tmem + ((32u * sp) << 16);

  const int ntiles = nk_tiles + nv_tiles;
  for (int tile = blockIdx.x; tile < ntiles && !failed; tile += gridDim.x) {
    const bool key = tile < nk_tiles;
    const QuantizeArgs& a = key ? ka : va;
    const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
    const long long gv = static_cast<long long>(key ? tile : tile - nk_tiles) * kRows + row;
    const bool valid = gv < nvec;
    const __nv_bfloat16* xrow = static_cast<const __nv_bfloat16*>(a.x) + gv * kD;

    // ---- 1. x quarter -> row statistics -> scaled fp16 tile ---------------
    uint4 raw[4];
    {
      const uint4* src = reinterpret_cast<const uint4*>(xrow + 32 * q);
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = valid ? src[c] : make_uint4(0u, 0u, 0u, 0u);
      float ss = 0.f, mx = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t wv[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(wv[k] << 16), hi = __uint_as_float(wv[k] & 0xFFFF0000u);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
          mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
        }
      }
      red_s[q * 128 + row] = ss;
      red_m[q * 128 + row] = mx;
    }
    __syncthreads();
    float nf, xs_scale = 1.0f, n16f;
    unsigned short n16;
    {
      const float ss = (red_s[row] + red_s[128 + row]) + (red_s[256 + row] + red_s[384 + row]);
      const float mx = fmaxf(fmaxf(red_m[row], red_m[128 + row]), fmaxf(red_m[256 + row], red_m[384 + row]));
      nf = sqrtf(ss);
      if (mx > 0.0f) {
        int e;
        frexpf(mx, &e);
        xs_scale = ldexpf(1.0f, 14 - e);
      }
      __half h = __float2half_rn(nf);
      const float hb = __half2float(h);
      const unsigned short hbits = __half_as_ushort(h);
      const float up = __half2float(__ushort_as_half(static_cast<unsigned short>(hbits + 1)));
      const float dn = hbits ? __half2float(__ushort_as_half(static_cast<unsigned short>(hbits - 1))) : 0.0f;
      const float tol = 4e-6f * nf;
      if (valid && nf > 0.0f && (fabsf(nf - 0.5f * (hb + up)) < tol || fabsf(nf - 0.5f * (hb + dn)) < tol)) {
        DF acc{0.f, 0.f};
        for (int k = 0; k < kD; ++k) {
          const float xv = __bfloat162float(xrow[k]);
          acc = df_add(acc, DF{xv * xv, 0.f});
        }
        const float r = sqrtf(acc.h);
        const float res = fmaf(-r, r, acc.h) + acc.l;
        const float rl2 = res / (2.0f * r);
        h = df_to_half(r + rl2, rl2 - ((r + rl2) - r));
      }
      n16 = __half_as_ushort(h);
      n16f = __half2float(h);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t wv[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
        uint32_t hv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 p = __floats2half2_rn(__uint_as_float(wv[k] << 16) * xs_scale,
                                              __uint_as_float(wv[k] & 0xFFFF0000u) * xs_scale);
          hv[k] = *reinterpret_cast<const uint32_t*>(&p);
        }
        *reinterpret_cast<uint4*>(smem + kOffX + swz_chunk(row, 4 * q + c, kRows)) =
            make_uint4(hv[0], hv[1], hv[2], hv[3]);
      }
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
      umma_commit(smem_u32(&bars[1]));
    }
    if (!mbar_wait(smem_u32(&bars[1]), phase)) {
      failed = true;
      if (tid == 0) atomicOr(a.tab.err, kErrTimeout);
    }
    phase ^= 1;
    tc_fence_after();

    // ---- 3. codes and residual of this quarter -------------------------------
    const int grp = q < 2 ? 0 : 1;
    const int gslot = (key ? 0 : 2) + grp;
    const float inv = 1.0f / (xs_scale * kPiScale);
    const float ku = nf > 0.0f ? inv * (kSqrtD / nf) : 0.0f;
    const float kr = n16f > 0.0f ? inv * (kSqrtD / n16f) : 0.0f;
    uint32_t words[4] = {0u, 0u, 0u, 0u};
    uint32_t rh[16], rl[16];
    uint32_t near = 0;
    float rho2 = 0.0f;
    {
      float v[32];
      tmem_ld32(trow + 32 * q, v);
      const Cell* cg = cells + gslot * kCells;
      const int bits = key ? (grp ? KBL : KBH) : (grp ? VBL : VBH);
      const float* cent = cents + gslot * 16;
      const double* t64 = t64s + gslot * 16;
      const int nb = (1 << bits) - 1;
      if (!valid) near = 0;
#define TQ_QUARTER(B, K)                                                                                       \
  do {                                                                                                         \
    quarter_epilogue<B, K>(v, cg, ku, kr, words, near, rho2, rh, rl);                                          \
    if (!valid) near = 0;                                                                                      \
    if (near)                                                                                                  \
      quarter_refine<B, K>(v, near, xrow, a.tab.pi_df, 32 * q, t64, nb, cent, kr, words, rho2, rh, rl,         \
                           &a.tab.counters[0]);                                                                \
  } while (0)
      if (key) {
        if (grp == 0) TQ_QUARTER(KBH, true);
        else TQ_QUARTER(KBL, true);
      } else {
        if (grp == 0) TQ_QUARTER(VBH, false);
        else TQ_QUARTER(VBL, false);
      }
#undef TQ_QUARTER
      if (key) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = swz_chunk(row, 4 * q + c, kRows);
          *reinterpret_cast<uint4*>(smem + kOffRH + off) = make_uint4(rh[4 * c], rh[4 * c + 1], rh[4 * c + 2], rh[4 * c + 3]);
          *reinterpret_cast<uint4*>(smem + kOffX + off) = make_uint4(rl[4 * c], rl[4 * c + 1], rl[4 * c + 2], rl[4 * c + 3]);
        }
        red_r[q * 128 + row] = rho2;
      }
    }

    // record location
    unsigned char* rec = nullptr;
    int slot = 0;
    if (valid) {
      const int h = static_cast<int>(gv % a.H);
      const long long bt = gv / a.H;
      const int t = static_cast<int>(bt % a.n_new);
      const int b = static_cast<int>(bt / a.n_new);
      const int pos = a.start_pos[b] + t;
      const int blk = pos >> 4;
      if (pos < 0 || blk >= a.maxp) {
        if (q == 0) atomicOr(a.tab.err, kErrBlock);
      } else {
        const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
        if (page < 0 || page >= a.num_pages) {
          if (q == 0) atomicOr(a.tab.err, kErrPage);
        } else {
          rec = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(h) * a.lay.block_bytes;
          slot = pos & 15;
        }
      }
    }
    if (rec) {
      const int bh = key ? KBH : VBH, bl = key ? KBL : VBL;
      const int woff = q < 2 ? q * bh : 2 * bh + (q - 2) * bl;
      const int nw = grp ? bl : bh;
      uint32_t* cw = reinterpret_cast<uint32_t*>(rec + slot * a.lay.code_bytes) + woff;
#pragma unroll
      for (int w = 0; w < 4; ++w)
        if (w < nw) cw[w] = words[w];
      if (q == 0) reinterpret_cast<unsigned short*>(rec + a.lay.off_norm)[slot] = n16;
    }

    // ---- 4. keys: z = r' S^T and the sign bits -------------------------------
    if (key) {
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
      if (!mbar_wait(smem_u32(&bars[1]), phase)) {
        failed = true;
        if (tid == 0) atomicOr(a.tab.err, kErrTimeout);
      }
      phase ^= 1;
      tc_fence_after();
      const float rho = sqrtf((red_r[row] + red_r[128 + row]) + (red_r[256 + row] + red_r[384 + row]));
      if (32 * q < m) {
        float v[32];
        tmem_ld32(trow + 128 + 32 * q, v);
        const float guard = kSignGuard * rho;
        uint32_t word = 0, nearz = 0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          word |= ((~__float_as_uint(v[k])) >> 31) << k;
          nearz |= (fabsf(v[k]) < guard ? 1u : 0u) << k;
        }
        if (!rec) nearz = 0;
        while (nearz) {
          const int k = __ffs(nearz) - 1;
          nearz &= nearz - 1;
          const int p = 32 * q + k;
          const uint32_t* cwr = reinterpret_cast<const uint32_t*>(rec + slot * a.lay.code_bytes);
          float cv[2 * kD];
          for (int j = 0; j < kD; ++j) {
            const int cj = record_code(cwr, KBH, KBL, j);
            const GroupBook& gb = a.lay.g[j < 64 ? 0 : 1];
            cv[2 * j] = gb.c[cj];
            cv[2 * j + 1] = gb.c_lo[cj];
          }
          const uint32_t bitv = refine_sign(xrow, a.tab.a_df + static_cast<long long>(p) * kD * 2,
                                            a.tab.s_df + static_cast<long long>(p) * kD * 2, cv, n16f);
          word = (word & ~(1u << k)) | (bitv << k);
          atomicAdd(&a.tab.counters[1], 1ULL);
        }
        if (rec) reinterpret_cast<uint32_t*>(rec + a.lay.off_signs + slot * (m / 8))[q] = word;
      }
      if (rec && q == 0)
        reinterpret_cast<unsigned short*>(rec + a.lay.off_rnorm)[slot] =
            __half_as_ushort(__float2half_rn(rho * n16f * kInvSqrtDHi));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int KBH, int KBL, int VBH, int VBL>
cudaError_t launch_tc(const QuantizeArgs& k, const QuantizeArgs& v, int nk, int nv, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(quantize_tc_kernel<KBH, KBL, VBH, VBL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes4);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = nk + nv;
  const int grid = tiles < sms ? tiles : sms;
  quantize_tc_kernel<KBH, KBL, VBH, VBL><<<grid, kThreadsTC4, kSmemBytes4, s>>>(k, v, nk, nv);
  return cudaGetLastError();
}

}  // namespace

bool launch_quantize_tc(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err) {
  const QuantizeArgs& any = k.x ? k : v;
  if (any.f32) return false;
  if ((k.x && (k.f32 || k.lay.split != 64 || k.m % 32 || k.m > 128 || !k.lay.qjl)) ||
      (v.x && (v.f32 || v.lay.split != 64)))
    return false;
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
