// Online quantize-and-append of bf16 K/V: a warp-specialized, pipelined
// tensor-core kernel (tcgen05 + TMA).
//
// [P2] "생각정리 209 (TurboQuant)", stage 1 and stage 2; [P4] riverfrot.github.io
// "TurboQuant란 무엇이며…", §4.1 (every vector is randomly rotated), §4.2 (the
// Lloyd-Max codebook is only looked up), §4.3 (residual r = x - Q^-1(Q(x)) and
// the 1-bit sign sketch of a random projection of r), §3.1 (paged blocks).
//
// One persistent CTA per SM, 18 warps, tiles of 128 vectors (K tiles first,
// then V tiles).  Roles:
//   warp 16, one lane: the TMA of x tiles (bf16 rows, two 64-channel boxes
//       with the 128-byte swizzle) into a two-stage ring, and every MMA:
//       y = x Pi^T as fp16 MMAs with Pi (scaled by 16) split into fp16 hi +
//       lo (about 22 bits) and x read from tensor memory; for keys, once r' is
//       written, z = r' S^T as three fp16 MMAs (r'_hi S_hi + r'_lo S_hi +
//       r'_hi S_lo) with r' read from tensor memory, into the columns y used;
//   warps 0-15: the epilogue, two groups of eight (group s takes the tiles of
//       slot s = local tile index % 2); a row (vector) has two threads, one
//       per 64-channel half: warp w reads tensor-memory lanes 32 (w % 4)..,
//       half (w / 4) % 2;
//   warp 17: the fixer.  A row whose fast path met a decision it cannot take
//       for certain (below) is handed to it through a shared-memory ring, and
//       it quantizes that vector again from x, every decision made exactly,
//       and rewrites the whole record.
// Tensor memory: slot s = columns [256 s, 256 s + 256): y, then z, in the first
// 128; in the second 128, first x (fp16, 64 columns), then r' (fp16 hi and
// lo, 64 columns each).  While one group works on tile j, the other group's
// tile and the TMA of tile j + 2 proceed.
//
// Epilogue of a tile, per thread (64 channels):
//   1. from the bf16 x tile in shared memory: the sum of squares of its half
//      (exact squares, fp32 sums), the halves added through shared memory, the
//      fp32 norm and its fp16 rounding; then x * 2^(14 - e), e the norm's
//      binary exponent, to fp16 (exact for bf16 values above 2^-28 of the
//      norm) into tensor memory for the y MMA.
//   2. per 32-channel chunk: fg = 8 u + 32, u = sqrt(d) y / ||x||; the cell
//      floor(fg) of a 128-entry table (cells of 1/8 over u in [-4, 12), the
//      unsigned conversion clamps the low end) gives the one boundary that can
//      matter there (in the same units) and the code below it; codes as
//      nibbles, then the stored words; for keys r' = y sqrt(d)/fp16(||x||) -
//      c[code] as fp16 hi + lo pairs stored to tensor memory.
//   3. keys: the sign bits of z; fp16(||r||) from the two halves' sums.
// The fast path writes every record.  A row goes to the fixer when its fp32
// norm lies within 4e-6 of an fp16 rounding midpoint, a u within 4.5e-6 of
// its boundary, or a |z| below 2e-5 ||r'||: after the group's next barrier
// (both halves have stored the row by then) its thread puts it in the ring.
// The fixer's own pass: the norm in double-float, y and z in fp32 with
// four partial sums, and every u within 1e-4 of a boundary or |z| within
// 2e-4 ||r|| of zero decided again in double-float.
// Every wait is bounded: a wait that gives up sets the error word and every
// later wait of that thread returns at once, so the CTA still reaches its end
// (every named barrier is still met).

#include "tq_internal.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

constexpr int kRows = 128;
constexpr int kEpiWarps = 16;
constexpr int kCtlWarp = 16;                 // TMA + MMA issue
constexpr int kFixWarp = 17;                 // exact re-quantization of flagged rows
constexpr int kThreadsP = (kEpiWarps + 2) * 32;
constexpr int kQueue = 64;                   // fixer ring entries (tile * 128 + row)
constexpr int kWaitLimitP = 1 << 22;
constexpr int kFixIdleLimit = 1 << 26;       // the fixer's polls of an empty ring (about 128 ns apart)
constexpr int kCells = 128;                  // cells of width 1/8 over u in [-4, 12)
constexpr float kSqrtD = 11.313708498984761f;
constexpr double kSqrtD64 = 11.313708498984760390;
constexpr float kInvSqrtDHi = 0.0883883461356163f;
constexpr float kInvSqrtDLo = 1.512702185735293e-09f;
// |u - t| < 4.5e-6 (in fg = 8u + 32 units): decide in double-float.  The fast u carries
// the 22-bit split of Pi, fp32 accumulation and norm (about 1e-7 typical) plus the
// rounding of fg and of the tabled 8t + 32 (2.4e-7 each).
constexpr float kGuardFg = 8.0f * 4.5e-6f;
constexpr float kGuardSign = 2e-5f;          // |z| < 2e-5 ||r'||: decide in double-float
// fp32 norm this close (relative) to an fp16 rounding midpoint: exact norm.  The
// sum of the (exact) squares rounds at most 8 times along any path, so its
// relative error is below 8 * 2^-24, the norm's below 3e-7.
constexpr float kNormTol = 5e-7f;
constexpr float kFixGuardU = 1e-4f;          // the fixer's fp32 u this close to a boundary: double-float
constexpr float kFixGuardZ = 2e-4f;          // the fixer's fp32 |z| below this times ||r||: double-float

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffPIH = 0;                   // 16 Pi rounded to fp16, 128 x 128, 128-byte swizzle, K-major
constexpr int kOffPIL = 32768;               // fp16(16 Pi - hi)
constexpr int kOffSH = 65536;                // S_hi fp16, m x 128
constexpr int kOffSL = 98304;                // S_lo
constexpr int kOffX = 131072;                // two bf16 x stages of 32 KB
constexpr int kOffTab = 196608;
// tables: per group (K hi, K lo, V hi, V lo)
constexpr int kTabCellT = 0;                 // [4][128] float 8 t + 32 of the cell's boundary
constexpr int kTabCellC = 2048;              // [4][128] int code below it
constexpr int kTabCent = 4096;               // [4][16] float centroids
constexpr int kTabCentLo = 4352;             // [4][16] float (c64 - c)
constexpr int kTabZero = 4608;               // [16] zeros (centroids of a zero-norm residual)
constexpr int kTabT64 = 4672;                // [4][16] double boundaries
constexpr int kTabSS = 5184;                 // [2 slots][2 halves][128] float
constexpr int kTabRho = 7232;                // [2][2][128] float
constexpr int kTabBar = 9280;                // mbarriers
constexpr int kBarTab = 0, kBarXFull = 1, kBarXFree = 3, kBarXTmem = 5, kBarYFull = 7, kBarRFull = 9, kBarZFull = 11,
              kNumBars = 13;
constexpr int kTabTmem = kTabBar + 8 * kNumBars;
constexpr int kTabT32 = kTabTmem + 16;       // [4][16] float boundaries (the fixer)
constexpr int kTabQ = kTabT32 + 256;         // the fixer's ring (32-bit words, below)
constexpr int kQTail = 0, kQHead = 1, kQDone = 2, kQProg = 4, kQVal = 8, kQSeq = 8 + 2 * kQueue;
constexpr int kQWords = kQSeq + kQueue;
constexpr int kTabBytes = kTabQ + 4 * kQWords;
constexpr int kSmemP = kOffTab + kTabBytes + 1024;
static_assert(kSmemP <= 232448, "shared memory per block");

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait; false (and nothing waited) once `failed` is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, bool& failed) {
  if (failed) return false;
  for (int i = 0; i < kWaitLimitP; ++i)
    if (mbar_test(bar, parity)) return true;
  failed = true;
  return false;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ float lds_f(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ int lds_i(uint32_t addr) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart; kdesc: k-step s (16 channels) of a 128-channel tile
// of `rows` rows (two 64-channel halves one after the other).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int s) {
  return sdesc(tile + (s >> 2) * rows * 128 + (s & 3) * 32);
}
// Instruction descriptor, kind::f16, fp32 accumulate, M = 128, N = n, K-major
// operands: bf16 (A and B) or fp16 (A and B); an A operand read from tensor
// memory holds row i in lane i, two 16-bit K values per 32-bit column.
__host__ __device__ constexpr uint32_t idesc(int n, bool bf16) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// ---------------------------------------------------------------------------
// double-float helpers (exact decisions)
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
__device__ __forceinline__ DF df_sq(float x) {
  const float p = x * x;
  return {p, fmaf(x, x, -p)};
}
__device__ __forceinline__ double df_to_d(DF a) { return static_cast<double>(a.h) + static_cast<double>(a.l); }
__device__ __forceinline__ DF warp_df_sum(DF v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    v = df_add(v, DF{__shfl_xor_sync(0xffffffffu, v.h, off), __shfl_xor_sync(0xffffffffu, v.l, off)});
  return v;
}
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
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// codes of a 32-channel chunk: first as plain 4-bit nibbles (channel c at bits
// 4 (c % 8) of word c / 8), then converted to the stored format (see tq.h),
// which fills exactly B consecutive words for the chunk
// ---------------------------------------------------------------------------
template <int POS>
__device__ __forceinline__ uint32_t bfi4(uint32_t base, uint32_t ins) {
  uint32_t d;
  asm("bfi.b32 %0, %1, %2, %3, 4;" : "=r"(d) : "r"(ins), "r"(base), "n"(POS));
  return d;
}
__device__ __forceinline__ uint32_t bfi4_dyn(uint32_t base, uint32_t ins, uint32_t pos) {
  uint32_t d;
  asm("bfi.b32 %0, %1, %2, %3, 4;" : "=r"(d) : "r"(ins), "r"(base), "r"(pos));
  return d;
}

// Stored words of a chunk from its nibble codes.
template <int B>
__device__ __forceinline__ void pack_words(const uint32_t (&cp)[4], uint32_t (&w)[4]) {
  if (B == 4) {
    // sign-magnitude: code >= 8 -> code - 8, else 15 - code, i.e. x ^ 8 ^ (7 if bit 3 clear)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lowmask = ((~cp[i]) & 0x88888888u) >> 3;
      w[i] = cp[i] ^ 0x88888888u ^ (lowmask * 7u);
    }
  } else if (B == 3) {
    // octets: channels 0-5 in the low 3 bits of nibbles 0-5, the bits of
    // channel 6 at 3/11/19 and of channel 7 at 7/15/23 (one multiply spreads
    // bit k of the two codes to 3 + 8k and 7 + 8k)
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = (cp[i] & 0x00777777u) | (((cp[i] >> 24) * 0x20408u) & 0x00888888u);
    w[0] = o[0] | (o[1] << 24);
    w[1] = (o[1] >> 8) | (o[2] << 16);
    w[2] = (o[2] >> 16) | (o[3] << 8);
    w[3] = 0u;
  } else if (B == 2) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t a = (cp[2 * i] | (cp[2 * i] >> 2)) & 0x0F0F0F0Fu;
      a = (a | (a >> 4)) & 0x00FF00FFu;
      a = (a | (a >> 8)) & 0x0000FFFFu;
      uint32_t b = (cp[2 * i + 1] | (cp[2 * i + 1] >> 2)) & 0x0F0F0F0Fu;
      b = (b | (b >> 4)) & 0x00FF00FFu;
      b = (b | (b >> 8)) & 0x0000FFFFu;
      w[i] = a | (b << 16);
    }
    w[2] = w[3] = 0u;
  } else {
    uint32_t acc = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t a = cp[i] & 0x11111111u;
      a = (a | (a >> 3)) & 0x03030303u;
      a = (a | (a >> 6)) & 0x000F000Fu;
      a = (a | (a >> 12)) & 0x000000FFu;
      acc |= a << (8 * i);
    }
    w[0] = acc;
    w[1] = w[2] = w[3] = 0u;
  }
}

__device__ __forceinline__ void pack_dispatch(int b, const uint32_t (&cp)[4], uint32_t (&w)[4]) {
  switch (b) {
    case 1: pack_words<1>(cp, w); break;
    case 2: pack_words<2>(cp, w); break;
    case 3: pack_words<3>(cp, w); break;
    default: pack_words<4>(cp, w); break;
  }
}

// Code of channel j (0..127) of a stored record (any bit width); reads go to L2.
__device__ int record_code(const uint32_t* cw, int bh, int bl, int split, int j) {
  const int grp = j < split ? 0 : 1, b = grp ? bl : bh, c = grp ? j - split : j, base = grp ? split * bh : 0;
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

// Cell of fg = 8u + 32: byte offset of its table entry (u < -4 clamps to 0).
__device__ __forceinline__ uint32_t cell_off(float fg) { return __float2uint_rd(fg) * 4u; }

// Pass A: codes of 16 channels (ctab: the group's cell boundaries as 8t + 32;
// ctab + 2048: the codes below them) as two nibble words, and the smallest
// |fg - t|.
__device__ __forceinline__ void codes_pass(const float (&v)[16], uint32_t ctab, float k8, uint32_t& cpa,
                                           uint32_t& cpb, float& dmin) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t word = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float fg = fmaf(v[8 * i + k], k8, 32.0f);
      const uint32_t off = cell_off(fg);
      const float t = lds_f(ctab + off);
      const int cl = lds_i(ctab + 2048u + off);
      const uint32_t code = static_cast<uint32_t>(cl + (fg >= t ? 1 : 0));
      dmin = fminf(dmin, fabsf(fg - t));
      switch (k) {
        case 0: word = code; break;
        case 1: word = bfi4<4>(word, code); break;
        case 2: word = bfi4<8>(word, code); break;
        case 3: word = bfi4<12>(word, code); break;
        case 4: word = bfi4<16>(word, code); break;
        case 5: word = bfi4<20>(word, code); break;
        case 6: word = bfi4<24>(word, code); break;
        default: word = bfi4<28>(word, code); break;
      }
    }
    if (i == 0) cpa = word;
    else cpb = word;
  }
}

// Pass B (keys): r' = y kr - c[code] for 16 channels (codes in cpa, cpb) as
// fp16 (hi, lo) pairs, and their sum of squares.
__device__ __forceinline__ void resid_pass(const float (&v)[16], uint32_t cpa, uint32_t cpb, uint32_t cent, float kr,
                                           float& rho2, uint32_t (&hi)[8], uint32_t (&lo)[8]) {
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t w = p < 4 ? cpa : cpb;
    const uint32_t code0 = (w >> (8 * (p & 3))) & 15u;
    const uint32_t code1 = (w >> (8 * (p & 3) + 4)) & 15u;
    const float r0 = fmaf(v[2 * p], kr, -lds_f(cent + code0 * 4u));
    const float r1 = fmaf(v[2 * p + 1], kr, -lds_f(cent + code1 * 4u));
    rho2 = fmaf(r0, r0, rho2);
    rho2 = fmaf(r1, r1, rho2);
    const __half2 h2 = __floats2half2_rn(r0, r1);
    const float2 hf = __half22float2(h2);
    const __half2 l2 = __floats2half2_rn(r0 - hf.x, r1 - hf.y);
    hi[p] = *reinterpret_cast<const uint32_t*>(&h2);
    lo[p] = *reinterpret_cast<const uint32_t*>(&l2);
  }
}

// x row (bf16, global memory): lane l takes channels 4l..4l+3.
__device__ __forceinline__ void lane_x(const __nv_bfloat16* xrow, int lane, float (&xv)[4]) {
  const uint2 r = reinterpret_cast<const uint2*>(xrow)[lane];
  xv[0] = bf16lo(r.x), xv[1] = bf16hi(r.x), xv[2] = bf16lo(r.y), xv[3] = bf16hi(r.y);
}

// Exact code of channel j (warp together, every lane returns it): y = Pi_j x
// and ||x||^2 in double-float, u = sqrt(d) y / ||x|| in double, compared with
// the fp64 boundaries.
__device__ __noinline__ int exact_code(const __nv_bfloat16* xrow, const float* pidf_row, const double* t64, int nb,
                                       int lane) {
  float xv[4];
  lane_x(xrow, lane, xv);
  const float4* pr = reinterpret_cast<const float4*>(pidf_row) + 2 * lane;
  const float4 p0 = __ldg(pr), p1 = __ldg(pr + 1);
  DF yd{0.f, 0.f}, n2{0.f, 0.f};
  yd = df_fma_acc(yd, p0.x, p0.y, xv[0]);
  yd = df_fma_acc(yd, p0.z, p0.w, xv[1]);
  yd = df_fma_acc(yd, p1.x, p1.y, xv[2]);
  yd = df_fma_acc(yd, p1.z, p1.w, xv[3]);
#pragma unroll
  for (int k = 0; k < 4; ++k) n2 = df_add(n2, df_sq(xv[k]));
  yd = warp_df_sum(yd);
  n2 = warp_df_sum(n2);
  const double n64 = sqrt(df_to_d(n2));
  const double u64 = n64 > 0.0 ? kSqrtD64 * df_to_d(yd) / n64 : 0.0;
  int code = 0;
  for (int k = 0; k < nb; ++k) code += u64 >= t64[k];
  return code;
}

// Exact sign bit of projection p (warp together): (S Pi)_p x - fp16(||x||)/sqrt(d) S_p c^ in double-float, with the
// codes read back from the stored record.
__device__ __noinline__ uint32_t exact_sign(const __nv_bfloat16* xrow, const float* adf_row, const float* sdf_row,
                                            const uint32_t* cw, int kbh, int kbl, int split, const float* cents,
                                            const float* centl, float n16f, int lane) {
  float xv[4];
  lane_x(xrow, lane, xv);
  const float4* ar = reinterpret_cast<const float4*>(adf_row) + 2 * lane;
  const float4* sr = reinterpret_cast<const float4*>(sdf_row) + 2 * lane;
  const float4 a0 = __ldg(ar), a1 = __ldg(ar + 1), s0 = __ldg(sr), s1 = __ldg(sr + 1);
  const float ah[4] = {a0.x, a0.z, a1.x, a1.z}, al[4] = {a0.y, a0.w, a1.y, a1.w};
  const float sh[4] = {s0.x, s0.z, s1.x, s1.z}, sl[4] = {s0.y, s0.w, s1.y, s1.w};
  DF d1{0.f, 0.f}, d2{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * lane + k;
    const int cj = record_code(cw, kbh, kbl, split, j) + (j < split ? 0 : 16);
    d1 = df_fma_acc(d1, ah[k], al[k], xv[k]);
    d2 = df_add(d2, df_mul(DF{sh[k], sl[k]}, DF{cents[cj], centl[cj]}));
  }
  d1 = warp_df_sum(d1);
  d2 = warp_df_sum(d2);
  const DF f = df_mul(DF{n16f, 0.f}, DF{kInvSqrtDHi, kInvSqrtDLo});
  const DF fz = df_mul(f, d2);
  const DF z = df_add(d1, DF{-fz.h, -fz.l});
  return (z.h > 0.0f || (z.h == 0.0f && z.l >= 0.0f)) ? 1u : 0u;
}

// Exact sign bit of projection p (warp together) from the lane's own four
// channels (4 lane .. 4 lane + 3): x and the centroid-table indices of their
// codes; the same double-float sum as exact_sign.
__device__ __noinline__ uint32_t exact_sign_regs(const float (&xv)[4], const float* adf_row, const float* sdf_row,
                                                 const int (&cidx)[4], const float* cents, const float* centl,
                                                 float n16f, int lane) {
  const float4* ar = reinterpret_cast<const float4*>(adf_row) + 2 * lane;
  const float4* sr = reinterpret_cast<const float4*>(sdf_row) + 2 * lane;
  const float4 a0 = __ldg(ar), a1 = __ldg(ar + 1), s0 = __ldg(sr), s1 = __ldg(sr + 1);
  const float ah[4] = {a0.x, a0.z, a1.x, a1.z}, al[4] = {a0.y, a0.w, a1.y, a1.w};
  const float sh[4] = {s0.x, s0.z, s1.x, s1.z}, sl[4] = {s0.y, s0.w, s1.y, s1.w};
  DF d1{0.f, 0.f}, d2{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    d1 = df_fma_acc(d1, ah[k], al[k], xv[k]);
    d2 = df_add(d2, df_mul(DF{sh[k], sl[k]}, DF{cents[cidx[k]], centl[cidx[k]]}));
  }
  d1 = warp_df_sum(d1);
  d2 = warp_df_sum(d2);
  const DF f = df_mul(DF{n16f, 0.f}, DF{kInvSqrtDHi, kInvSqrtDLo});
  const DF fz = df_mul(f, d2);
  const DF z = df_add(d1, DF{-fz.h, -fz.l});
  return (z.h > 0.0f || (z.h == 0.0f && z.l >= 0.0f)) ? 1u : 0u;
}

// Record of vector gv (null when its position or page is out of range; the
// epilogue flags those).
__device__ __forceinline__ unsigned char* locate(const QuantizeArgs& a, long long gv, long long nvec, int& slot,
                                                 bool flag) {
  int hh, t, b;
  if (nvec < (1LL << 31)) {
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
    if (flag) atomicOr(a.tab.err, kErrBlock);
    return nullptr;
  }
  const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
  if (page < 0 || page >= a.num_pages) {
    if (flag) atomicOr(a.tab.err, kErrPage);
    return nullptr;
  }
  slot = pos & 15;
  return a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(hh) * a.lay.block_bytes;
}

__device__ __forceinline__ uint32_t ld_vol(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}
__device__ __forceinline__ void st_vol(uint32_t* p, uint32_t v) { *reinterpret_cast<volatile uint32_t*>(p) = v; }

// The fixer's ring (one producer thread at a time per call): reserve n
// consecutive entries if there is room (false: decide here instead), then
// write each entry and publish it by its sequence number.  An entry is two
// words: local tile index << 7 | row, and kind << 16 | channel or projection.
__device__ bool ring_reserve(uint32_t* q, uint32_t n, uint32_t& base) {
  for (int it = 0; it < 64; ++it) {
    const uint32_t t = ld_vol(q + kQTail);
    if (t + n - ld_vol(q + kQHead) > static_cast<uint32_t>(kQueue)) return false;
    if (atomicCAS(q + kQTail, t, t + n) == t) {
      base = t;
      return true;
    }
  }
  return false;
}
__device__ __forceinline__ void ring_publish(uint32_t* q, uint32_t idx, uint32_t v0, uint32_t v1) {
  st_vol(q + kQVal + 2 * (idx % kQueue), v0);
  st_vol(q + kQVal + 2 * (idx % kQueue) + 1, v1);
  __threadfence_block();
  st_vol(q + kQSeq + idx % kQueue, idx + 1);
}
constexpr uint32_t kEntryCode = 0u, kEntrySign = 1u;

// 8 bits to bits 0, 4, ..., 28.
__device__ __forceinline__ uint32_t spread4(uint32_t x) {
  x = (x | (x << 12)) & 0x000F000Fu;
  x = (x | (x << 6)) & 0x03030303u;
  return (x | (x << 3)) & 0x11111111u;
}

// The fixer: quantize vector gv again (the whole warp; lane l owns channels
// and projections 4l .. 4l + 3) with every decision exact, and rewrite its
// record: fp16 norm from a double-float norm; y = Pi x in fp32 (four partial
// sums of 32 terms); codes, the ones within kFixGuardU of a boundary decided
// in double-float; keys: r = y - fp16(||x||)/sqrt(d) c[code], z = S r in fp32,
// the |z| below kFixGuardZ ||r|| decided in double-float; fp16(||r||).
__device__ __forceinline__ void fix_vector(const QuantizeArgs& a, bool key, bool qjl, long long gv, long long nvec,
                                           const unsigned char* tab, int bits0, int bits1, int split, int lane) {
  int slot = 0;
  unsigned char* rec = locate(a, gv, nvec, slot, false);
  if (!rec) return;                                         // warp-uniform
  const __nv_bfloat16* xrow = static_cast<const __nv_bfloat16*>(a.x) + gv * kD;
  const int gofs = key ? 0 : 2;
  float xv[4];
  lane_x(xrow, lane, xv);
  DF n2{0.f, 0.f};
#pragma unroll
  for (int k = 0; k < 4; ++k) n2 = df_add(n2, df_sq(xv[k]));
  n2 = warp_df_sum(n2);
  float nf = 0.0f;
  __half n16h = __float2half_rn(0.0f);
  if (n2.h > 0.0f) {
    const float rr = sqrtf(n2.h);
    const float rl = (fmaf(-rr, rr, n2.h) + n2.l) / (2.0f * rr);
    nf = rr + rl;
    n16h = df_to_half(nf, rl - (nf - rr));
  }
  const float n16f = __half2float(n16h);

  // y = Pi x: x_k from lane k / 4, row k of Pi^T (fp32) as one float4 per lane
  float y[4];
  {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c][i] = 0.0f;
    const float4* pt = reinterpret_cast<const float4*>(a.tab.pit) + lane;
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float xk = __shfl_sync(0xffffffffu, xv[c], k >> 2);
        const float4 p4 = __ldg(pt + (k + c) * (kD / 4));
        acc[c][0] = fmaf(p4.x, xk, acc[c][0]);
        acc[c][1] = fmaf(p4.y, xk, acc[c][1]);
        acc[c][2] = fmaf(p4.z, xk, acc[c][2]);
        acc[c][3] = fmaf(p4.w, xk, acc[c][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
  }

  // codes
  const float* t32 = reinterpret_cast<const float*>(tab + kTabT32);
  const double* t64 = reinterpret_cast<const double*>(tab + kTabT64);
  const float ku = nf > 0.0f ? kSqrtD / nf : 0.0f;
  int code[4];
  uint32_t pend = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = 4 * lane + i, grp = j < split ? 0 : 1, nb = (1 << (grp ? bits1 : bits0)) - 1;
    const float u = y[i] * ku;
    const float* tb = t32 + (gofs + grp) * 16;
    int c = 0;
    bool near = false;
    for (int k = 0; k < nb; ++k) {
      c += u >= tb[k] ? 1 : 0;
      near = near || fabsf(u - tb[k]) < kFixGuardU;
    }
    code[i] = c;
    pend |= (near ? 1u : 0u) << i;
  }
  for (int it = 0; it < 128; ++it) {                         // at most 4 per lane: 128 rounds
    const uint32_t who = __ballot_sync(0xffffffffu, pend != 0u);
    if (!who) break;
    const int src = __ffs(who) - 1;
    const int i = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
    if (lane == src) pend &= pend - 1u;
    const int j = 4 * src + i, grp = j < split ? 0 : 1, nb = (1 << (grp ? bits1 : bits0)) - 1;
    const int c = exact_code(xrow, a.tab.pi_df + j * kD * 2, t64 + (gofs + grp) * 16, nb, lane);
    if (lane == src) code[i] = c;
  }

  // stored code words: channels 8w .. 8w + 7 as nibbles come from lanes 2w, 2w + 1
  uint32_t* cw = reinterpret_cast<uint32_t*>(rec + slot * a.lay.code_bytes);
  {
    const uint32_t nib = static_cast<uint32_t>(code[0] | (code[1] << 4) | (code[2] << 8) | (code[3] << 12));
    const uint32_t pairw = nib | (__shfl_down_sync(0xffffffffu, nib, 1) << 16);
    uint32_t cp[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cp[i] = __shfl_sync(0xffffffffu, pairw, (lane & ~7) + 2 * i);
    if ((lane & 7) == 0) {
      const int ch0 = 4 * lane, grp = ch0 < split ? 0 : 1, b = grp ? bits1 : bits0;
      uint32_t w[4];
      pack_dispatch(b, cp, w);
      uint32_t* dst = cw + ((grp ? split * bits0 : 0) + (ch0 - grp * split) * b) / 32;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k < b) dst[k] = w[k];
    }
  }
  if (lane == 0) *(reinterpret_cast<unsigned short*>(rec + a.lay.off_norm) + slot) = __half_as_ushort(n16h);
  if (!(key && qjl)) return;

  // residual, its norm, z = S r
  const float* cents = reinterpret_cast<const float*>(tab + kTabCent);
  const float* centl = reinterpret_cast<const float*>(tab + kTabCentLo);
  const float cs = n16f * kInvSqrtDHi;
  float r[4];
  int cidx[4];
  float rho2 = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = 4 * lane + i;
    cidx[i] = (j < split ? 0 : 16) + code[i];
    r[i] = n16f > 0.0f ? fmaf(-cs, cents[cidx[i]], y[i]) : y[i];
    rho2 = fmaf(r[i], r[i], rho2);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) rho2 += __shfl_xor_sync(0xffffffffu, rho2, o);
  const float rho = sqrtf(rho2);
  const int m = a.m;
  const bool own = 4 * lane < m;
  float z[4];
  {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c][i] = 0.0f;
    const float4* st4 = reinterpret_cast<const float4*>(a.tab.st) + (own ? lane : 0);
#pragma unroll 2
    for (int j = 0; j < kD; j += 4) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float rj = __shfl_sync(0xffffffffu, r[c], j >> 2);
        const float4 s4 = __ldg(st4 + (j + c) * (m / 4));
        acc[c][0] = fmaf(s4.x, rj, acc[c][0]);
        acc[c][1] = fmaf(s4.y, rj, acc[c][1]);
        acc[c][2] = fmaf(s4.z, rj, acc[c][2]);
        acc[c][3] = fmaf(s4.w, rj, acc[c][3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) z[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
  }
  uint32_t sb = 0u;
  pend = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sb |= (z[i] >= 0.0f ? 1u : 0u) << i;
    pend |= (own && fabsf(z[i]) < kFixGuardZ * rho ? 1u : 0u) << i;
  }
  for (int it = 0; it < 128; ++it) {
    const uint32_t who = __ballot_sync(0xffffffffu, pend != 0u);
    if (!who) break;
    const int src = __ffs(who) - 1;
    const int i = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
    if (lane == src) pend &= pend - 1u;
    const int p = 4 * src + i;
    const uint32_t bit = exact_sign_regs(xv, a.tab.a_df + static_cast<long long>(p) * kD * 2,
                                         a.tab.s_df + static_cast<long long>(p) * kD * 2, cidx, cents, centl, n16f, lane);
    if (lane == src) sb = (sb & ~(1u << i)) | (bit << i);
  }
  // sign word w: bit 4 (l - 8w) + i is projection 4l + i
  uint32_t bl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) bl[i] = __ballot_sync(0xffffffffu, (sb >> i) & 1u);
  if (lane < m / 32) {
    uint32_t word = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) word |= spread4((bl[i] >> (8 * lane)) & 0xFFu) << i;
    reinterpret_cast<uint32_t*>(rec + a.lay.off_signs + slot * (m / 8))[lane] = word;
  }
  if (lane == 0)
    *(reinterpret_cast<unsigned short*>(rec + a.lay.off_rnorm) + slot) = __half_as_ushort(__float2half_rn(rho));
}

// Cell table of one group: cell g covers u in [-4 + g/8, -4 + (g+1)/8) (cell 0
// reaches down to -inf, cell 127 up to +inf); it keeps the boundary inside it,
// else the nearest one (as 8t + 32), and the number of boundaries below that
// boundary.  Boundaries are >= 1/4 apart, so u one cell off by rounding still
// gets the right code or lies within the guard of that boundary.
__device__ void build_cell(float* cell_t, int* cell_c, const GroupBook& gb, int g) {
  const float lo = -4.0f + g * 0.125f, hi = lo + 0.125f;
  int inside = -1, nearest = 0;
  float best = INFINITY;
  for (int k = 0; k < gb.nb; ++k) {
    const float t = gb.t[k];
    const bool in = (t >= lo || g == 0) && (t < hi || g == kCells - 1);
    if (in && inside < 0) inside = k;
    const float dist = t < lo ? lo - t : (t >= hi ? t - hi : 0.0f);
    if (dist < best) { best = dist; nearest = k; }
  }
  const int k = inside >= 0 ? inside : nearest;
  cell_t[g] = fmaf(gb.t[k], 8.0f, 32.0f);
  cell_c[g] = k;
}

struct PipeParams {
  int nk, nv;                 // K tiles, V tiles
  int kbits[2], vbits[2];     // per channel group
  int ksplit, vsplit;
};

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// 18 warps need <= 96 registers a thread: five warps share one SM sub-partition.
__global__ void __maxnreg__(96)
    quantize_pipe_kernel(QuantizeArgs ka, QuantizeArgs va, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, PipeParams pp) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t tabs = sb + kOffTab;
  unsigned char* tab = smem + kOffTab;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = pp.nk + pp.nv;
  const int m = ka.m;
  const bool kqjl = pp.nk > 0 && ka.lay.qjl;
  auto bar = [&](int i) { return tabs + kTabBar + 8u * static_cast<uint32_t>(i); };

  // ---- tables, barriers, tensor memory ------------------------------------
  for (int i = tid; i < 4 * kCells; i += kThreadsP) {
    const int grp = i / kCells;
    const GroupBook& gb = (grp < 2 ? ka.lay : va.lay).g[grp & 1];
    build_cell(reinterpret_cast<float*>(tab + kTabCellT) + grp * kCells,
               reinterpret_cast<int*>(tab + kTabCellC) + grp * kCells, gb, i % kCells);
  }
  if (tid < 64) {
    const int grp = tid >> 4, k = tid & 15;
    const GroupBook& gb = (grp < 2 ? ka.lay : va.lay).g[grp & 1];
    reinterpret_cast<float*>(tab + kTabCent)[tid] = k < (1 << gb.bits) ? gb.c[k] : 0.0f;
    reinterpret_cast<float*>(tab + kTabCentLo)[tid] = k < (1 << gb.bits) ? gb.c_lo[k] : 0.0f;
    reinterpret_cast<double*>(tab + kTabT64)[tid] = gb.t64[k];
    reinterpret_cast<float*>(tab + kTabT32)[tid] = k < gb.nb ? gb.t[k] : 0.0f;
    if (tid < 16) reinterpret_cast<float*>(tab + kTabZero)[tid] = 0.0f;
  }
  for (int i = tid; i < kQWords; i += kThreadsP) reinterpret_cast<uint32_t*>(tab + kTabQ)[i] = 0u;
  if (warp == kCtlWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tabs + kTabTmem),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(bar(kBarTab), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarXFull + s), 1);
      mbar_init(bar(kBarXFree + s), 8);
      mbar_init(bar(kBarXTmem + s), 8);
      mbar_init(bar(kBarYFull + s), 1);
      mbar_init(bar(kBarRFull + s), 8);
      mbar_init(bar(kBarZFull + s), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async();
    const uint32_t bytes = 2 * 32768 + (kqjl ? 2 * m * 256 : 0);
    mbar_arrive_tx(bar(kBarTab), bytes);
    bulk_g2s(sb + kOffPIH, ka.tab.pih_sw, 32768, bar(kBarTab));
    bulk_g2s(sb + kOffPIL, ka.tab.pil_sw, 32768, bar(kBarTab));
    if (kqjl) {
      bulk_g2s(sb + kOffSH, ka.tab.sh_sw, m * 256, bar(kBarTab));
      bulk_g2s(sb + kOffSL, ka.tab.sl_sw, m * 256, bar(kBarTab));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(tab + kTabTmem);
  bool failed = false;
  auto tile_of = [&](int j) { return static_cast<int>(blockIdx.x) + j * static_cast<int>(gridDim.x); };
  int local_tiles = 0;
  if (static_cast<int>(blockIdx.x) < ntiles)
    local_tiles = (ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;

  if (warp == kCtlWarp) {
    // ---- TMA and MMA issue (one lane), in the order their inputs become ready
    if (lane == 0) {
      bool ok = mbar_wait(bar(kBarTab), 0, failed);
      tc_fence_after();
      int nx = 0, ny = 0, nz = 0, idle = 0;
      while (ok && nz < local_tiles) {
        bool progressed = false;
        // TMA of tile nx into stage nx % 2 once the epilogue released it
        if (nx < local_tiles && (nx < 2 || mbar_test(bar(kBarXFree + (nx & 1)), ((nx - 2) >> 1) & 1))) {
          const int st = nx & 1;
          const int tile = tile_of(nx);
          const bool key = tile < pp.nk;
          const int row0 = (key ? tile : tile - pp.nk) * kRows;
          const CUtensorMap* map = key ? &tmk : &tmv;
          mbar_arrive_tx(bar(kBarXFull + st), 2 * 16384);
          tma_2d(sb + kOffX + st * 32768, map, 0, row0, bar(kBarXFull + st));
          tma_2d(sb + kOffX + st * 32768 + 16384, map, 64, row0, bar(kBarXFull + st));
          ++nx;
          progressed = true;
        }
        // z of tile nz (keys) once its residual is in tensor memory
        if (nz < ny) {
          const bool key = tile_of(nz) < pp.nk;
          if (!key || !kqjl) {
            ++nz;
            progressed = true;
          } else if (mbar_test(bar(kBarRFull + (nz & 1)), (nz >> 1) & 1)) {
            tc_fence_after();
            const int s = nz & 1;
            const uint32_t zt = tmem + 256u * s;                 // over the consumed y
            const uint32_t rh = tmem + 256u * s + 128u, rl = rh + 64u;
            const uint32_t id = idesc(m, false);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              umma_ts(zt, rh + 8u * t, kdesc(sb + kOffSH, m, t), id, t > 0);
              umma_ts(zt, rl + 8u * t, kdesc(sb + kOffSH, m, t), id, 1u);
              umma_ts(zt, rh + 8u * t, kdesc(sb + kOffSL, m, t), id, 1u);
            }
            umma_commit(bar(kBarZFull + s));
            ++nz;
            progressed = true;
          }
        }
        // y of tile ny once the epilogue wrote its fp16 x to tensor memory
        // (which it does only after it finished the slot's previous tile)
        if (ny < local_tiles && ny < nz + 2 && mbar_test(bar(kBarXTmem + (ny & 1)), (ny >> 1) & 1)) {
          tc_fence_after();
          const int s = ny & 1;
          const uint32_t yt = tmem + 256u * s, xt = tmem + 256u * s + 128u;
          const uint32_t id = idesc(128, false);
#pragma unroll
          for (int t = 0; t < 8; ++t) umma_ts(yt, xt + 8u * t, kdesc(sb + kOffPIH, kRows, t), id, t > 0);
#pragma unroll
          for (int t = 0; t < 8; ++t) umma_ts(yt, xt + 8u * t, kdesc(sb + kOffPIL, kRows, t), id, 1u);
          umma_commit(bar(kBarYFull + s));
          ++ny;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > kWaitLimitP) {
          failed = true;
          ok = false;
        }
      }
      if (failed) atomicOr(ka.tab.err, kErrTimeout);
      // copies and MMAs still in flight complete before the CTA ends
      bool f2 = false;
      for (int j = (nx >= 2 ? nx - 2 : 0); j < nx; ++j) (void)mbar_wait(bar(kBarXFull + (j & 1)), (j >> 1) & 1, f2);
      if (ny > 0) (void)mbar_wait(bar(kBarYFull + ((ny - 1) & 1)), ((ny - 1) >> 1) & 1, f2);
      if (nz > 0 && kqjl && tile_of(nz - 1) < pp.nk)
        (void)mbar_wait(bar(kBarZFull + ((nz - 1) & 1)), ((nz - 1) >> 1) & 1, f2);
    }
    __syncwarp();
  } else if (warp == kFixWarp) {
    // ---- fixer: decisions from the ring until both epilogue groups are done ---------
    // A code entry: the exact code, compared with the stored one; when they differ
    // (the fast path was wrong, not just close) the row is quantized again as a
    // whole, once the group is past it.  A sign entry: the exact sign bit, patched
    // into the stored word.
    uint32_t* q = reinterpret_cast<uint32_t*>(tab + kTabQ);
    const float* cents_k = reinterpret_cast<const float*>(tab + kTabCent);
    const float* centl_k = reinterpret_cast<const float*>(tab + kTabCentLo);
    uint32_t h = 0;
    int idle = 0;
    for (;;) {
      uint32_t v0 = 0u, v1 = 0u, have = 0u;
      if (lane == 0 && ld_vol(q + kQSeq + h % kQueue) == h + 1) {
        __threadfence_block();
        v0 = ld_vol(q + kQVal + 2 * (h % kQueue));
        v1 = ld_vol(q + kQVal + 2 * (h % kQueue) + 1);
        have = 1u;
      }
      have = __shfl_sync(0xffffffffu, have, 0);
      if (have) {
        v0 = __shfl_sync(0xffffffffu, v0, 0);
        v1 = __shfl_sync(0xffffffffu, v1, 0);
        ++h;
        if (lane == 0) st_vol(q + kQHead, h);                 // the entry is free again
        idle = 0;
        const int jl = static_cast<int>(v0 >> 7), row = static_cast<int>(v0 & 127u);
        const int tile = tile_of(jl);
        const bool key = tile < pp.nk;
        const QuantizeArgs& a = key ? ka : va;
        const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
        const long long gv = static_cast<long long>(key ? tile : tile - pp.nk) * kRows + row;
        const int bits0 = key ? pp.kbits[0] : pp.vbits[0], bits1 = key ? pp.kbits[1] : pp.vbits[1];
        const int split = key ? pp.ksplit : pp.vsplit;
        int slot = 0;
        unsigned char* rec = locate(a, gv, nvec, slot, false);
        if (!rec) continue;
        const __nv_bfloat16* sx = static_cast<const __nv_bfloat16*>(a.x) + gv * kD;
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(rec + slot * a.lay.code_bytes);
        const int idx = static_cast<int>(v1 & 0xFFFFu);
        if ((v1 >> 16) == kEntryCode) {
          const int grp = idx < split ? 0 : 1;
          const int code = exact_code(sx, a.tab.pi_df + idx * kD * 2,
                                      reinterpret_cast<const double*>(tab + kTabT64) + ((key ? 0 : 2) + grp) * 16,
                                      (1 << (grp ? bits1 : bits0)) - 1, lane);
          if (lane == 0) atomicAdd(&a.tab.counters[0], 1ULL);
          if (code != record_code(cw, bits0, bits1, split, idx)) {
            // the rest of the row depends on this code: wait until the group
            // is past the row's tile, then quantize the vector again
            bool ok = false;
            for (int it = 0; it < kWaitLimitP && !ok; ++it) {
              ok = static_cast<int>(ld_vol(q + kQProg + (jl & 1))) > jl;
              if (!ok) __nanosleep(64);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1u : 0u, 0) != 0u;
            if (!ok) {
              failed = true;
              break;
            }
            __threadfence();
            fix_vector(a, key, kqjl, gv, nvec, tab, bits0, bits1, split, lane);
          }
        } else {
          const float n16f = __half2float(__ushort_as_half(
              __ldcg(reinterpret_cast<const unsigned short*>(rec + a.lay.off_norm) + slot)));
          const uint32_t bit = exact_sign(sx, a.tab.a_df + static_cast<long long>(idx) * kD * 2,
                                          a.tab.s_df + static_cast<long long>(idx) * kD * 2, cw, bits0, bits1, split,
                                          cents_k, centl_k, n16f, lane);
          if (lane == 0) {
            atomicAdd(&a.tab.counters[1], 1ULL);
            uint32_t* sw = reinterpret_cast<uint32_t*>(rec + a.lay.off_signs + slot * (a.m / 8)) + idx / 32;
            const uint32_t w = __ldcg(sw), nw = (w & ~(1u << (idx & 31))) | (bit << (idx & 31));
            if (nw != w) *sw = nw;
          }
        }
        __syncwarp();
        continue;
      }
      uint32_t done = 0u;
      if (lane == 0 && ld_vol(q + kQDone) == 2u) {
        __threadfence_block();
        done = ld_vol(q + kQTail) == h ? 1u : 0u;
      }
      if (__shfl_sync(0xffffffffu, done, 0)) break;
      if (++idle > kFixIdleLimit) {
        failed = true;
        break;
      }
      __nanosleep(128);
    }
    if (failed && lane == 0) atomicOr(ka.tab.err, kErrTimeout);
  } else {
    // ---- epilogue ---------------------------------------------------------------
    const int q = warp & 3, h = (warp >> 2) & 1, s = warp >> 3;
    const int row = 32 * q + lane;
    const int gbar = 1 + s;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + 256u * s;
    float* ss_part = reinterpret_cast<float*>(tab + kTabSS) + s * 256;
    float* rho_part = reinterpret_cast<float*>(tab + kTabRho) + s * 256;
    const float* cents_k = reinterpret_cast<const float*>(tab + kTabCent);
    const float* centl_k = reinterpret_cast<const float*>(tab + kTabCentLo);
    uint32_t* qring = reinterpret_cast<uint32_t*>(tab + kTabQ);
    for (int j = s; j < local_tiles; j += 2) {
      const int tile = tile_of(j);
      const bool key = tile < pp.nk;
      const QuantizeArgs& a = key ? ka : va;
      const int par = (j >> 1) & 1;
      const long long nvec = static_cast<long long>(a.batch) * a.n_new * a.H;
      const long long gv0 = static_cast<long long>(key ? tile : tile - pp.nk) * kRows;
      const bool valid = gv0 + row < nvec;
      const bool sk = key && kqjl;
      const int split = key ? pp.ksplit : pp.vsplit;
      const int bits0 = key ? pp.kbits[0] : pp.vbits[0], bits1 = key ? pp.kbits[1] : pp.vbits[1];

      // ---- 1. norm, fp16 x into tensor memory ------------------------------------
      (void)mbar_wait(bar(kBarXFull + s), par, failed);
      const unsigned char* xt = smem + kOffX + s * 32768 + h * 16384 + row * 128;
      {
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(xt + ((c ^ (row & 7)) << 4));
          const float x0 = bf16lo(w4.x), x1 = bf16hi(w4.x), x2 = bf16lo(w4.y), x3 = bf16hi(w4.y);
          const float x4 = bf16lo(w4.z), x5 = bf16hi(w4.z), x6 = bf16lo(w4.w), x7 = bf16hi(w4.w);
          float a0 = x0 * x0;
          a0 = fmaf(x1, x1, a0);
          a0 = fmaf(x2, x2, a0);
          a0 = fmaf(x3, x3, a0);
          float a1 = x4 * x4;
          a1 = fmaf(x5, x5, a1);
          a1 = fmaf(x6, x6, a1);
          a1 = fmaf(x7, x7, a1);
          acc[c] = a0 + a1;
        }
        ss_part[h * 128 + row] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
      named_sync(gbar, 256);
      // the group is past its previous tile (the fixer may rewrite those rows)
      if (q == 0 && h == 0 && lane == 0) st_vol(qring + kQProg + s, static_cast<uint32_t>(j));
      const float ss = ss_part[row] + ss_part[128 + row];
      float nf = ss > 0.0f ? sqrtf(ss) : 0.0f;
      // x * 2^(14 - e) with nf < 2^e: every |x_k| <= ||x|| stays below 2^14
      float xs = 1.0f;
      if (nf > 0.0f) {
        int e;
        frexpf(nf, &e);
        xs = ldexpf(1.0f, 14 - e);
      }
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {          // 32 channels (16 columns) at a time, re-read from the x tile
        uint32_t hx[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(xt + (((4 * hq + c) ^ (row & 7)) << 4));
          const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __half2 p2 = __floats2half2_rn(bf16lo(ww[k]) * xs, bf16hi(ww[k]) * xs);
            hx[4 * c + k] = *reinterpret_cast<const uint32_t*>(&p2);
          }
        }
        tmem_st16(trow + 128u + 32u * h + 16u * hq, hx);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarXTmem + s));      // the y MMA may start
      __half n16h = __float2half_rn(nf);
      bool near_mid = false;
      if (nf > 0.0f) {
        const float hb = __half2float(n16h);
        const unsigned short hbits = __half_as_ushort(n16h);
        const float up = __half2float(__ushort_as_half(static_cast<unsigned short>(hbits + 1)));
        const float dn = hbits ? __half2float(__ushort_as_half(static_cast<unsigned short>(hbits - 1))) : 0.0f;
        const float tol = kNormTol * nf;
        near_mid = fabsf(nf - 0.5f * (hb + up)) < tol || fabsf(nf - 0.5f * (hb + dn)) < tol;
      }
      // exact norm of the flagged rows, the warp together (both halves' warps do
      // the same and get the same value)
      uint32_t nm = __ballot_sync(0xffffffffu, near_mid);
      while (nm) {
        const int src = __ffs(nm) - 1;
        nm &= nm - 1;
        const int r = 32 * q + src;
        const int k = 4 * lane;
        const unsigned char* xr = smem + kOffX + s * 32768 + (k >> 6) * 16384 + r * 128;
        const uint2 w2 = *reinterpret_cast<const uint2*>(xr + ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
        DF n2 = df_add(df_add(df_sq(bf16lo(w2.x)), df_sq(bf16hi(w2.x))), df_add(df_sq(bf16lo(w2.y)), df_sq(bf16hi(w2.y))));
        n2 = warp_df_sum(n2);
        if (lane == src) {
          const float rr = sqrtf(n2.h);
          const float rl = (fmaf(-rr, rr, n2.h) + n2.l) / (2.0f * rr);
          nf = rr + rl;
          n16h = df_to_half(nf, rl - (nf - rr));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarXFree + s));        // this warp is done with the x tile
      const float n16f = __half2float(n16h);
      // y from the MMA is 16 xs y: fg = 8 u + 32 = y_mma k8 + 32
      const float ku = nf > 0.0f ? kSqrtD / (nf * xs * 16.0f) : 0.0f;
      const float k8 = 8.0f * ku;
      // a zero fp16 norm leaves the residual equal to y scaled (any positive
      // scale gives the same signs): formed without the centroids
      const float kr = n16f > 0.0f ? kSqrtD / (n16f * xs * 16.0f) : ku;

      // record location of this row
      unsigned char* rec = nullptr;
      int slot = 0;
      if (valid) {
        const long long gv = gv0 + row;
        int hh, t, b;
        if (nvec < (1LL << 31)) {
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
          if (h == 0) atomicOr(a.tab.err, kErrBlock);
        } else {
          const int page = a.block_table[static_cast<long long>(b) * a.maxp + blk];
          if (page < 0 || page >= a.num_pages) {
            if (h == 0) atomicOr(a.tab.err, kErrPage);
          } else {
            rec = a.cache + static_cast<long long>(page) * a.page_bytes + static_cast<long long>(hh) * a.lay.block_bytes;
            slot = pos & 15;
          }
        }
      }
      uint32_t* const cw = rec ? reinterpret_cast<uint32_t*>(rec + slot * a.lay.code_bytes) : nullptr;

      // ---- 2. codes and residual --------------------------------------------------
      (void)mbar_wait(bar(kBarYFull + s), par, failed);
      tc_fence_after();
      float rho2 = 0.0f;
      const int gofs = key ? 0 : 2;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int ch0 = 64 * h + 32 * c;                 // first channel of the chunk
        const int grp = ch0 < split ? 0 : 1;
        const int b = grp ? bits1 : bits0;
        const uint32_t ctab = tabs + kTabCellT + (gofs + grp) * kCells * 4;
        uint32_t cp[4];
        uint32_t dpend[2] = {0u, 0u}, dbase[2] = {0u, 0u};   // codes handed to the fixer
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {               // 16 channels at a time (rolled: a smaller loop body
                                                        // for the instruction cache, 2% faster at c2)
          const int cb = ch0 + 16 * hh;
          float v[16];
          tmem_ld16(trow + cb, v);
          uint32_t cpa, cpb;
          float dmin = INFINITY;
          codes_pass(v, ctab, k8, cpa, cpb, dmin);
          if (!valid || nf == 0.0f || !cw) dmin = INFINITY;
          // rare: codes within the guard of their boundary go to the fixer (published
          // once this chunk's words are stored); when its ring has no room, the warp
          // decides them here and patches their nibbles
          uint32_t pend = 0u;
          if (dmin < kGuardFg) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const float fg = fmaf(v[cc], k8, 32.0f);
              pend |= (fabsf(fg - lds_f(ctab + cell_off(fg))) < kGuardFg ? 1u : 0u) << cc;
            }
            if (ring_reserve(qring, __popc(pend), dbase[hh])) {
              dpend[hh] = pend;
              pend = 0u;
            }
          }
          if (__any_sync(0xffffffffu, pend != 0u)) {
            for (;;) {
              const uint32_t who = __ballot_sync(0xffffffffu, pend != 0);
              if (!who) break;
              const int src = __ffs(who) - 1;
              const int cc = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
              if (lane == src) pend &= pend - 1;
              const __nv_bfloat16* sx = static_cast<const __nv_bfloat16*>(a.x) + (gv0 + 32 * q + src) * kD;
              const int code = exact_code(sx, a.tab.pi_df + (cb + cc) * kD * 2,
                                          reinterpret_cast<const double*>(tab + kTabT64) + (gofs + grp) * 16,
                                          (1 << b) - 1, lane);
              if (lane == 0) atomicAdd(&a.tab.counters[0], 1ULL);
              if (lane == src) {
                const uint32_t nb = static_cast<uint32_t>(code), pos = 4u * (cc & 7);
                if (cc < 8) cpa = bfi4_dyn(cpa, nb, pos);
                else cpb = bfi4_dyn(cpb, nb, pos);
              }
            }
          }
          if (sk) {
            const uint32_t cent = (n16f > 0.0f) ? tabs + kTabCent + (gofs + grp) * 64 : tabs + kTabZero;
            uint32_t hi[8], lo[8];
            resid_pass(v, cpa, cpb, cent, kr, rho2, hi, lo);
            tmem_st8(trow + 128u + (cb >> 1), hi);
            tmem_st8(trow + 192u + (cb >> 1), lo);
          }
          cp[2 * hh] = cpa;
          cp[2 * hh + 1] = cpb;
        }
        if (cw) {
          // the chunk's b words: channels ch0.. of group grp start at stream bit
          // (grp ? split * bits0 : 0) + (ch0 - grp * split) * b, a word boundary
          uint32_t w[4];
          pack_dispatch(b, cp, w);
          uint32_t* dst = cw + ((grp ? split * bits0 : 0) + (ch0 - grp * split) * b) / 32;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k < b) dst[k] = w[k];
        }
        if (dpend[0] | dpend[1]) {
          __threadfence();                               // the words are stored before the fixer reads them
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pm = dpend[hh], idx = dbase[hh];
            while (pm) {
              const int cc = __ffs(pm) - 1;
              pm &= pm - 1u;
              ring_publish(qring, idx++, (static_cast<uint32_t>(j) << 7) | static_cast<uint32_t>(row),
                           (kEntryCode << 16) | static_cast<uint32_t>(ch0 + 16 * hh + cc));
            }
          }
        }
      }
      if (h == 0 && rec) *(reinterpret_cast<unsigned short*>(rec + a.lay.off_norm) + slot) = __half_as_ushort(n16h);
      if (sk) {
        rho_part[h * 128 + row] = rho2;
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarRFull + s));
        named_sync(gbar, 256);                           // both halves' codes and residual sums are in
        const float rho = sqrtf(rho_part[row] + rho_part[128 + row]);
        // ---- 3. signs ----------------------------------------------------------------
        (void)mbar_wait(bar(kBarZFull + s), par, failed);
        tc_fence_after();
        const int nzc = m / 32, c0 = h ? (nzc + 1) / 2 : 0, c1 = h ? nzc : (nzc + 1) / 2;
        const float guard = kGuardSign * rho;
        uint32_t* const sgn = rec ? reinterpret_cast<uint32_t*>(rec + a.lay.off_signs + slot * (m / 8)) : nullptr;
        for (int c = c0; c < c1; ++c) {
          float v[32];
          tmem_ld32(trow + 32u * c, v);
          uint32_t neg = 0;
          float amin = INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            neg |= (__float_as_uint(v[k]) >> 31) << k;
            amin = fminf(amin, fabsf(v[k]));
          }
          uint32_t word = ~neg;
          if (!sgn) amin = INFINITY;
          // rare: signs of |z| within the guard go to the fixer after the word is
          // stored, or (no room in its ring) are decided here by the warp
          uint32_t pend = 0u, dp = 0u, db = 0u;
          if (amin <= guard) {
#pragma unroll
            for (int k = 0; k < 32; ++k) pend |= (fabsf(v[k]) <= guard ? 1u : 0u) << k;
            if (ring_reserve(qring, __popc(pend), db)) {
              dp = pend;
              pend = 0u;
            }
          }
          if (__any_sync(0xffffffffu, pend != 0u)) {
            for (;;) {
              const uint32_t who = __ballot_sync(0xffffffffu, pend != 0);
              if (!who) break;
              const int src = __ffs(who) - 1;
              const int kk = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
              if (lane == src) pend &= pend - 1;
              const __nv_bfloat16* sx = static_cast<const __nv_bfloat16*>(a.x) + (gv0 + 32 * q + src) * kD;
              const uint32_t* scw = reinterpret_cast<const uint32_t*>(__shfl_sync(
                  0xffffffffu, reinterpret_cast<unsigned long long>(cw), src));
              const float sn16 = __shfl_sync(0xffffffffu, n16f, src);
              const int p = 32 * c + kk;
              const uint32_t bit = exact_sign(sx, a.tab.a_df + static_cast<long long>(p) * kD * 2,
                                              a.tab.s_df + static_cast<long long>(p) * kD * 2, scw, bits0, bits1,
                                              split, cents_k, centl_k, sn16, lane);
              if (lane == 0) atomicAdd(&a.tab.counters[1], 1ULL);
              if (lane == src) word = (word & ~(1u << kk)) | (bit << kk);
            }
          }
          if (sgn) sgn[c] = word;
          if (dp) {
            __threadfence();
            while (dp) {
              const int kk = __ffs(dp) - 1;
              dp &= dp - 1u;
              ring_publish(qring, db++, (static_cast<uint32_t>(j) << 7) | static_cast<uint32_t>(row),
                           (kEntrySign << 16) | static_cast<uint32_t>(32 * c + kk));
            }
          }
        }
        if (h == 0 && rec)
          *(reinterpret_cast<unsigned short*>(rec + a.lay.off_rnorm) + slot) =
              __half_as_ushort(__float2half_rn(rho * n16f * kInvSqrtDHi));
      }
      tc_fence_before();
    }
    // every row of this group is stored and every entry published: tell the fixer
    named_sync(gbar, 256);
    if (q == 0 && h == 0 && lane == 0) {
      st_vol(qring + kQProg + s, 0x7FFFFFFFu);
      __threadfence_block();
      atomicAdd(qring + kQDone, 1u);
    }
    if (failed) atomicOr(ka.tab.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kCtlWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                                     : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Tensor map of a bf16 [nvec][128] input: boxes of 64 channels x 128 rows,
// 128-byte swizzle, rows past the end read as zeros.
bool make_map(CUtensorMap* map, const void* x, long long nvec) {
  auto fn = encode_fn();
  if (!fn || nvec < 1) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(nvec)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, kRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The cell tables need boundaries at least two cells (1/4) apart, inside (-3.875, 3.875).
bool cells_ok(const GroupBook& g) {
  for (int k = 0; k < g.nb; ++k) {
    if (!(g.t[k] > -3.875f && g.t[k] < 3.875f)) return false;
    if (k > 0 && g.t[k] - g.t[k - 1] < 0.25f) return false;
  }
  return true;
}

}  // namespace

bool launch_quantize_pipe(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err) {
  const QuantizeArgs& any = k.x ? k : v;
  if (any.f32) return false;
  if ((k.x && (k.m % 32 || k.m < 32 || k.m > 128)) || (k.x && k.lay.split % 32) || (v.x && v.lay.split % 32))
    return false;
  if ((reinterpret_cast<uintptr_t>(k.x) | reinterpret_cast<uintptr_t>(v.x)) & 15) return false;
  for (int g = 0; g < 2; ++g)
    if ((k.x && (!cells_ok(k.lay.g[g]) || k.lay.g[g].bits > 4)) || (v.x && (!cells_ok(v.lay.g[g]) || v.lay.g[g].bits > 4)))
      return false;
  const long long nk_vec = k.x ? static_cast<long long>(k.batch) * k.n_new * k.H : 0;
  const long long nv_vec = v.x ? static_cast<long long>(v.batch) * v.n_new * v.H : 0;
  const long long tiles = (nk_vec + kRows - 1) / kRows + (nv_vec + kRows - 1) / kRows;
  if (tiles < 1 || tiles > (1LL << 30)) return false;
  CUtensorMap mk, mv;
  if (k.x && !make_map(&mk, k.x, nk_vec)) return false;
  if (v.x && !make_map(&mv, v.x, nv_vec)) return false;
  if (!k.x) mk = mv;
  if (!v.x) mv = mk;
  PipeParams pp{};
  pp.nk = static_cast<int>((nk_vec + kRows - 1) / kRows);
  pp.nv = static_cast<int>((nv_vec + kRows - 1) / kRows);
  const KindLayout& kl = k.x ? k.lay : v.lay;
  const KindLayout& vl = v.x ? v.lay : k.lay;
  pp.kbits[0] = kl.g[0].bits, pp.kbits[1] = kl.g[1].bits;
  pp.vbits[0] = vl.g[0].bits, pp.vbits[1] = vl.g[1].bits;
  pp.ksplit = kl.split, pp.vsplit = vl.split;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = smem_attr_once(quantize_pipe_kernel, kSmemP, configured);
  if (e != cudaSuccess) { *err = e; return true; }
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int cap = any.max_ctas > 0 && any.max_ctas < sms ? any.max_ctas : sms;
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  if ((tiles + grid - 1) / grid >= (1LL << 24)) return false;   // ring entries hold a CTA's tile index in 25 bits
  const QuantizeArgs& kk = k.x ? k : v;
  const QuantizeArgs& vv = v.x ? v : k;
  quantize_pipe_kernel<<<grid, kThreadsP, kSmemP, s>>>(kk, vv, mk, mv, pp);
  *err = cudaGetLastError();
  return true;
}

}  // namespace tq
