// Multi-query causal attention over the compressed cache on the tensor cores
// (tcgen05): a block of 128 query rows against 64-token tiles of the cache,
// flash-style, with the cache dequantized once per block instead of once per
// eight rows.
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.3 (every new token's
// K/V join the cache; new token t's query attends over its prefix), §4.3 (the
// score: stage-1 reconstruction plus the QJL correction; softmax(score·scale)),
// §4.2 (the codebook is only looked up); [P2] "생각정리 209 (TurboQuant)", stage 2.
//
// An item is (sequence b, KV head h, block of 128 query rows r = t·G + g,
// chunk of key positions).  Per 64-token tile, with base-2 logits:
//   S = Q~ K^T + U A'^T   (one accumulator: M = 128 rows, N = 64 tokens)
//       Q~ = hi + lo fp16 and U = S·Pi q in fp16 sit in tensor memory;
//       K^ = the key's centroids and A' = (fb_t/fa_t)(2 b − 1) from the sign
//       bits, fp16 in shared memory, with fa_t = n_t/sqrt(d) and fb_t =
//       sqrt(pi/2)/m·rho_t;
//   logit = scale·log2(e)·fa_t·S + bias_t, bias_t = −∞ for a token that is
//       not there (past the tile or on a skipped page), −∞ too past the row's
//       causal end;
//   online softmax per row (the running max moves only when a logit passes it
//   by more than 3, so p ≤ 8 fits fp16);
//   [O | l] += P [V' | 1]  (P = p as fp16 in tensor memory; V' = n_v/sqrt(d)
//       times the values' centroids, token rows in shared memory read MN-major,
//       with a column of ones beside it so that column 128 accumulates the
//       softmax sum: M = 128, N = 144, K = 64 tokens).
// Each item ends with the chunk partial (max, sum, O) of its 128 rows; the
// decode's merge kernel combines the chunks and rotates back.
//
// One persistent CTA per SM, 18 warps:
//   warp 0: items from a global counter; a tile's four K and V page blocks by
//       bulk copy into a three-stage ring (page ids of the item loaded once);
//   warp 1: tensor memory (496 of 512 columns) and, one lane, the MMAs;
//   warps 4, 5, 16, 17: K^ rows and the token factors (two buffers, free again
//       once the tile's S MMAs have run);
//   warps 2, 3, 6, 7: the sign rows A' (in the K buffers, as soon as S of two
//       tiles back has run), then V' rows and the ones column (two buffers,
//       free again once the tile's O MMAs have run);
//   (a warp runs on SMSP warp % 4: each SMSP holds two softmax warps and one
//   side of the operand work, so that fewer code paths share its instruction
//   cache)
//   warps 8-15: the softmax.  Warps w and w + 4 share tensor-memory lanes
//       32 (w % 4) .. + 31, thread = query row; the first takes tokens 0-31
//       of a tile, the second 32-63, and they agree on the row max through
//       shared memory.
// Every wait is bounded; a wait that gives up sets the device error word and
// the CTA still reaches its end.

#include "tq_internal.h"
#include "tq_tc.cuh"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>
#include <utility>

namespace tq {
namespace {

using namespace tcx;

constexpr int kCR = 128;                  // query rows per item (MMA M)
constexpr int kCT = 64;                   // tokens per tile
constexpr int kCMaxChunk = 1024;          // an item's page ids: two per lane of a warp
constexpr int kCOpWarps = 8, kCEpWarps = 8;
constexpr int kCThreadsTC = 32 * (2 + kCOpWarps + kCEpWarps);
constexpr int kCStages = 3;
constexpr long long kCPollLimit = 1LL << 26;   // idle polls of the MMA lane before it gives up
constexpr int kCVN = 144;                 // V' columns: 128 channels, the ones column, 15 zero columns
constexpr float kInvSqrtDC = 0.08838834764831845f;
constexpr float kSqrtHalfPiC = 1.2533141373155003f;
constexpr float kLazyC = 3.0f;
constexpr float kNegBigC = -1.0e30f;
// tensor-memory columns
constexpr uint32_t kTQH = 0, kTQL = 64, kTU = 128, kTS = 192, kTO = 320, kTP = 480;
static_assert(kTO + kCVN <= kTP && kTP + 32 <= 512, "tensor memory columns");

// Lookup table of the fp16 centroid pair of a byte of two codes, per bit width
// (replicated per lane: entry e at 128 e + 4 lane), at these offsets.
__host__ __device__ constexpr int lut_entries_c(int b) { return b == 4 ? 256 : b == 3 ? 120 : 16; }
constexpr int kLut2 = 0, kLut3 = 16 * 128, kLut4 = kLut3 + 120 * 128, kLutBytes = kLut4 + 256 * 128;
__host__ __device__ constexpr int lut_off(int b) { return b == 4 ? kLut4 : b == 3 ? kLut3 : kLut2; }
__device__ __forceinline__ int stored_code_c(int b, int f) { return b == 4 ? (f < 8 ? f + 8 : 15 - f) : f; }

struct CDesc {                 // one tile of the stream
  int item;                    // -1: end
  int tile, last, first;
  int p0, npos;                // first position, positions in the tile (<= 64)
  unsigned mask;               // valid pages (4 bits)
  int b, h, qb, chunk;         // the item: sequence, KV head, query block, chunk
  int start;                   // the sequence's first new position
  int pad[4];
};
static_assert(sizeof(CDesc) == 64, "descriptor size");

template <int KBH, int KBL, int VBH, int VBL, bool QJL>
struct CGeo {
  static constexpr int CBK = 8 * (KBH + KBL);
  static constexpr int CBV = 8 * (VBH + VBL);
  static constexpr int KBB = 16 * (CBK + (QJL ? 16 + 2 : 0) + 2);
  static constexpr int VBB = 16 * (CBV + 2);
  static constexpr int K_SIGNS = 16 * CBK;
  static constexpr int K_NORM = K_SIGNS + (QJL ? 16 * 16 : 0);
  static constexpr int K_RNORM = K_NORM + 32;
  static constexpr int V_NORM = 16 * CBV;
  static constexpr int PAGE = KBB + VBB;           // a page: K block, then V block
  static constexpr int STAGE = 4 * PAGE;           // a tile
  // shared memory (offsets from a 1024-aligned base)
  // in an operand buffer: K^ and A' [64 tokens][128] K-major, V' [64 tokens][192] MN-major (three
  // 64-channel blocks of [64][128 B]; the third holds the ones column and zeros)
  static constexpr int KH = 0, AS = 16384, VT = 32768;
  static constexpr int OPS_BYTES = VT + 3 * 64 * 128;
  static constexpr int OPS = 0;
  static constexpr int LUT = OPS + 2 * OPS_BYTES;
  static constexpr int SGN = LUT + kLutBytes;      // sign masks of a nibble: [16][32 lanes] x 8 bytes
  static constexpr int REC = SGN + 16 * 32 * 8;
  static constexpr int FAC = (REC + kCStages * STAGE + 1023) & ~1023;   // [4][fa | bias][64] floats
  static constexpr int XMAX = FAC + 4 * 2 * 64 * 4;                     // [2][2][128] partial row maxima
  static constexpr int DESC = XMAX + 2 * 2 * 128 * 4;                   // [4] CDesc + [kCStages] CDesc
  static constexpr int BAR = DESC + (4 + kCStages) * 64;
  static constexpr int kRecFull = 0, kRecEmpty = 3, kKOps = 6, kVOps = 8, kKFree = 10, kVFree = 12,
                       kDescFull = 14, kSFull = 18, kSEmpty = 19, kPFull = 20, kODone = 21, kQReady = 22,
                       kDrain = 23, kXch = 24, kNumBar = 32;  // kXch + 2 q + parity: the row-max exchange of pair q
  static constexpr int TMEMA = BAR + 8 * kNumBar;
  static constexpr int SMEM = TMEMA + 16 + 1024;
  static_assert(KBB % 16 == 0 && VBB % 16 == 0, "bulk copy unit");
  static_assert(OPS_BYTES % 1024 == 0, "operand tiles on 1024-byte boundaries");
  static_assert(SMEM <= 232448, "shared memory per block");
};

__device__ __forceinline__ uint32_t octet_nibbles_c(uint32_t v) {
  return (v & 0x00777777u) | (((v & 0x00888888u) * 0x00204080u) & 0x77000000u);
}
__device__ __forceinline__ uint32_t stream_bits_c(const uint32_t (&w)[17], int off) {
  return (off & 31) ? __funnelshift_r(w[off >> 5], w[(off >> 5) + 1], off & 31) : w[off >> 5];
}
// Lookup indices of chunk cc (8 channels) of a group of B-bit codes at stream
// bit `base`: byte i = the index of channels (2i, 2i + 1).
template <int B>
__device__ __forceinline__ uint32_t chunk_bytes_c(const uint32_t (&w)[17], int base, int cc) {
  if (B == 4) return w[(base >> 5) + cc];
  if (B == 3) return octet_nibbles_c(stream_bits_c(w, base + 24 * cc));
  const uint32_t x = stream_bits_c(w, base + 16 * cc) & 0xFFFFu;
  return (x & 0xFu) | ((x & 0xF0u) << 4) | ((x & 0xF00u) << 8) | ((x & 0xF000u) << 12);
}
// Lookup indices of chunk cc (8 channels) of a 64-channel group of B-bit codes
// at `src` (8 B bytes): byte i = the index of channels (2i, 2i + 1).  The words
// are loaded first (chunk_words) so that two chunks' loads are in flight
// together, then unpacked (chunk_index).
template <int B>
__device__ __forceinline__ uint2 chunk_words(uint32_t src, int cc) {
  const int off = B * 8 * cc, wi = off >> 5, sh = off & 31;
  return make_uint2(lds32(src + 4 * wi), (B == 3 && sh > 8) ? lds32(src + 4 * wi + 4) : 0u);
}
template <int B>
__device__ __forceinline__ uint32_t chunk_index(uint2 w, int cc) {
  const int sh = (B * 8 * cc) & 31;
  if (B == 4) return w.x;
  if (B == 3) return octet_nibbles_c(sh ? __funnelshift_r(w.x, w.y, sh) : w.x);
  const uint32_t y = (w.x >> sh) & 0xFFFFu;
  return (y & 0xFu) | ((y & 0xF0u) << 4) | ((y & 0xF00u) << 8) | ((y & 0xF000u) << 12);
}

// Rows of one 64-channel half for token row t (B-bit codes at `src`): the fp16
// centroid pair of every channel pair, times f2 when SCALE (V'), zero for an
// invalid token.  Two chunks per step with their loads ahead of their stores
// (the shared-memory accesses keep program order); the step loop stays rolled
// because the kernel's roles share each SM's instruction cache.
template <int B, bool SCALE>
__device__ __forceinline__ void half_rows(uint32_t tile, uint32_t src, int t, int hf, bool tv, uint32_t tb,
                                          __half2 f2) {
#pragma unroll 1
  for (int cc = 0; cc < 8; cc += 2) {
    uint32_t p[2][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};
    if (tv) {
      const uint2 w0 = chunk_words<B>(src, cc), w1 = chunk_words<B>(src, cc + 1);
      const uint32_t x0 = chunk_index<B>(w0, cc), x1 = chunk_index<B>(w1, cc + 1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        p[0][i] = lds32(tb + __byte_perm(x0, 0u, 0x4440u + i) * 128u);
        p[1][i] = lds32(tb + __byte_perm(x1, 0u, 0x4440u + i) * 128u);
      }
      if (SCALE) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&p[j][i]), f2);
            p[j][i] = *reinterpret_cast<const uint32_t*>(&r);
          }
      }
    }
    sts128(tile + chunk_off(t, 8 * hf + cc, kCT), p[0][0], p[0][1], p[0][2], p[0][3]);
    sts128(tile + chunk_off(t, 8 * hf + cc + 1, kCT), p[1][0], p[1][1], p[1][2], p[1][3]);
  }
}

// 2^x by the SFU (ex2.approx.ftz: relative error about 2^-22; -inf gives 0).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory descriptor of an MN-major operand with 128-byte swizzle: rows
// of 64 MN elements (128 B) along K, 8-row groups 1024 B apart, 64-element MN
// blocks 8192 B apart.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(8192 >> 4) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

template <int KBH, int KBL, int VBH, int VBL, bool QJL>
__global__ void __launch_bounds__(kCThreadsTC, 1)
    causal_tc_kernel(const __grid_constant__ DecodeArgs a, int total_items, int nqb) {
  using G = CGeo<KBH, KBL, VBH, VBL, QJL>;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((0u - su32(sm_raw)) & 1023u);
  const uint32_t sb = su32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto barx = [&](int i) { return sb + G::BAR + 8u * static_cast<uint32_t>(i); };
  const int nch = a.nchunks, C = a.chunk, rows_all = a.T * a.G;
  auto seq_len = [&](int b) {
    int L = a.seq_lens[b] + a.len_add;
    if (L < 0 || L > a.max_seq_len || L > a.maxp * kPage) {
      atomicOr(a.tab.err, kErrSeqLen);
      L = L < 0 ? 0 : L;
      L = L > a.max_seq_len ? a.max_seq_len : L;
      L = L > a.maxp * kPage ? a.maxp * kPage : L;
    }
    return L;
  };
  // item -> (b, h, query block, chunk) and its key range [c0, c1): the chunk
  // cut at the causal end of the block's last row
  auto item_range = [&](int it, int& b, int& h, int& qb, int& chunk, int& c0, int& c1) {
    chunk = it % nch;
    const int rest = it / nch;
    qb = rest % nqb;
    const int bh = rest / nqb;
    h = bh % a.H;
    b = bh / a.H;
    const int last_row = min(rows_all, kCR * (qb + 1)) - 1;
    const int Lq = min(seq_len(b), a.seq_lens[b] + last_row / a.G + 1);
    c0 = chunk * C;
    c1 = min(c0 + C, Lq);
  };

  // ---- setup: lookup tables, the constant rows of V'^, barriers, tensor memory ------
  {
    for (int i = tid; i < kLutBytes / 4; i += kCThreadsTC) {
      const int off = 4 * i;
      const int b = off >= kLut4 ? 4 : off >= kLut3 ? 3 : 2;
      const int e = (off - lut_off(b)) >> 7;
      const int w = b == 2 ? 2 : 4, mask = b == 4 ? 15 : b == 3 ? 7 : 3;
      const int ilo = stored_code_c(b, e & mask), ihi = stored_code_c(b, (e >> w) & mask);
      // one codebook per bit width (the host checks that the groups agree)
      float clo = 0.0f, chi = 0.0f;
      bool has = true;
      if (a.kl.g[0].bits == b) {
        clo = a.kl.g[0].c[ilo];
        chi = a.kl.g[0].c[ihi];
      } else if (a.kl.g[1].bits == b) {
        clo = a.kl.g[1].c[ilo];
        chi = a.kl.g[1].c[ihi];
      } else if (a.vl.g[0].bits == b) {
        clo = a.vl.g[0].c[ilo];
        chi = a.vl.g[0].c[ihi];
      } else if (a.vl.g[1].bits == b) {
        clo = a.vl.g[1].c[ilo];
        chi = a.vl.g[1].c[ihi];
      } else {
        has = false;
      }
      uint32_t v = 0u;
      if (has && e < lut_entries_c(b))
        v = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(clo))) |
            (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(chi))) << 16);
      *reinterpret_cast<uint32_t*>(sm + G::LUT + off) = v;
    }
    // nibble n of sign bits (projections 4j .. 4j + 3) -> two words of fp16 sign masks: the sign
    // of a half is set where the bit is clear (2 b - 1 = -1)
    for (int i = tid; i < 16 * 32; i += kCThreadsTC) {
      const int n = i >> 5;
      const uint32_t w0 = ((n & 1) ? 0u : 0x8000u) | ((n & 2) ? 0u : 0x80000000u);
      const uint32_t w1 = ((n & 4) ? 0u : 0x8000u) | ((n & 8) ? 0u : 0x80000000u);
      *reinterpret_cast<uint2*>(sm + G::SGN + 8 * i) = make_uint2(w0, w1);
    }
    if (tid == 0) {
      for (int s = 0; s < kCStages; ++s) {
        bar_init(barx(G::kRecFull + s), 1);
        bar_init(barx(G::kRecEmpty + s), kCOpWarps);
      }
      for (int s = 0; s < 2; ++s) {
        bar_init(barx(G::kKOps + s), kCOpWarps);      // K^ rows (K side) and A' rows (V side)
        bar_init(barx(G::kVOps + s), kCOpWarps / 2);
        bar_init(barx(G::kKFree + s), 1);
        bar_init(barx(G::kVFree + s), 1);
      }
      for (int s = 0; s < 4; ++s) bar_init(barx(G::kDescFull + s), kCOpWarps / 2);
      bar_init(barx(G::kSFull), 1);
      bar_init(barx(G::kSEmpty), kCEpWarps);
      bar_init(barx(G::kPFull), kCEpWarps);
      bar_init(barx(G::kODone), 1);
      bar_init(barx(G::kQReady), kCEpWarps);
      bar_init(barx(G::kDrain), 1);
      for (int q = 0; q < 8; ++q) bar_init(barx(G::kXch + q), 2);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + G::TMEMA), "r"(512)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_wait();                        // the query prep before this kernel zeroed the counter and wrote q~/u
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
  }
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(sm + G::TMEMA);
  bool failed = false;
  CDesc* desc = reinterpret_cast<CDesc*>(sm + G::DESC);                // per tile of the stream (4)
  CDesc* rec_desc = reinterpret_cast<CDesc*>(sm + G::DESC + 4 * 64);   // per record stage

  if (warp == 0) {
    // ---- producer: items, page ids, the tile's page blocks ----------------------------
    int seq = 0, item = -1, ntile = 0, tile = 0, b = 0, h = 0, qb = 0, chunk = 0, c0 = 0, c1 = 0;
    int pid0 = -1, pid1 = -1;            // page ids 2 lane, 2 lane + 1 of the item (from page c0 / 16)
    for (;; ++seq) {
      const int s = seq % kCStages;
      bool ok = true;
      if (lane == 0 && seq >= kCStages)
        ok = bar_wait(barx(G::kRecEmpty + s), (seq / kCStages - 1) & 1, failed);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        failed = true;
        break;
      }
      while (item != -2 && tile >= ntile) {          // the next item with work
        int it = 0;
        if (lane == 0) it = atomicAdd(a.sched, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        if (it >= total_items) {
          item = -2;
          break;
        }
        item_range(it, b, h, qb, chunk, c0, c1);
        if (c1 <= c0) continue;
        item = it;
        tile = 0;
        ntile = (c1 - c0 + kCT - 1) / kCT;
        const int pg0 = c0 >> 4, npg = (c1 - 1) / 16 - pg0 + 1;
        const int* row = a.block_table + static_cast<long long>(b) * a.maxp + pg0;
        pid0 = 2 * lane < npg ? __ldg(row + 2 * lane) : -1;
        pid1 = 2 * lane + 1 < npg ? __ldg(row + 2 * lane + 1) : -1;
      }
      CDesc d{};
      d.item = -1;
      if (item >= 0) {
        d.item = item;
        d.tile = tile;
        d.first = tile == 0;
        d.last = tile == ntile - 1;
        d.p0 = c0 + kCT * tile;
        d.npos = min(kCT, c1 - d.p0);
        d.b = b;
        d.h = h;
        d.qb = qb;
        d.chunk = chunk;
        d.start = a.seq_lens[b];
      }
      // the tile's pages: lane j < 4 takes page j of the tile
      const int pg = (d.item >= 0 ? (d.p0 - c0) >> 4 : 0) + (lane & 3);
      const int v0 = __shfl_sync(0xffffffffu, pid0, (pg >> 1) & 31), v1 = __shfl_sync(0xffffffffu, pid1, (pg >> 1) & 31);
      const int pid = (pg & 1) ? v1 : v0;
      const bool in_range = d.item >= 0 && lane < 4 && 16 * lane < d.npos;
      const bool valid = in_range && pid >= 0 && pid < a.num_pages;
      if (in_range && !valid) atomicOr(a.tab.err, kErrPage);
      const uint32_t mask = __ballot_sync(0xffffffffu, valid);
      d.mask = mask;
      if (lane == 0) {
        rec_desc[s] = d;
        if (mask) bar_arrive_tx(barx(G::kRecFull + s), static_cast<uint32_t>(__popc(mask) * G::PAGE));
        else bar_arrive(barx(G::kRecFull + s));
      }
      __syncwarp();
      if (valid) {
        fence_async_smem();
        const uint32_t dst = sb + G::REC + s * G::STAGE + lane * G::PAGE;
        g2s(dst, a.kc + static_cast<long long>(pid) * a.k_page_bytes + static_cast<long long>(h) * G::KBB, G::KBB,
            barx(G::kRecFull + s));
        g2s(dst + G::KBB, a.vc + static_cast<long long>(pid) * a.v_page_bytes + static_cast<long long>(h) * G::VBB,
            G::VBB, barx(G::kRecFull + s));
      }
      if (d.item < 0) break;
      ++tile;
    }
    if (lane == 0) {                                 // copies still in flight land before the CTA ends
      bool f2 = false;
      for (int j = seq >= kCStages ? seq - kCStages + 1 : 0; j <= seq; ++j)
        (void)bar_wait(barx(G::kRecFull + j % kCStages), (j / kCStages) & 1, f2);
    }
  } else if (warp == 1) {
    // ---- MMA issue: the whole warp runs the loop converged (branch conditions are warp
    // votes) and one elected lane issues each MMA and commit, so that the operands stay in
    // uniform registers --------------------------------------------------------------------
    constexpr uint32_t id_s = idesc_f16(kCT), id_o = idesc_f16(kCVN) | (1u << 16);   // O: B MN-major
    auto uni = [](bool x) { return __all_sync(0xffffffffu, x); };
    auto issue_s = [&](int k) {
      const uint32_t kh = sb + G::OPS + (k & 1) * G::OPS_BYTES + G::KH, as = kh - G::KH + G::AS;
      tc_after();
#pragma unroll
      for (int j = 0; j < 8; ++j) mma_ts_warp(tmem + kTS, tmem + kTQH + 8u * j, kdesc(kh, kCT, j), id_s, j > 0 ? 1u : 0u);
#pragma unroll
      for (int j = 0; j < 8; ++j) mma_ts_warp(tmem + kTS, tmem + kTQL + 8u * j, kdesc(kh, kCT, j), id_s, 1u);
      if (QJL) {
#pragma unroll
        for (int j = 0; j < 8; ++j) mma_ts_warp(tmem + kTS, tmem + kTU + 8u * j, kdesc(as, kCT, j), id_s, 1u);
      }
      mma_commit_warp(barx(G::kSFull));
      mma_commit_warp(barx(G::kKFree + (k & 1)));
    };
    auto issue_o = [&](int k, bool first) {
      const uint32_t vt = sb + G::OPS + (k & 1) * G::OPS_BYTES + G::VT;
      tc_after();
#pragma unroll
      for (int j = 0; j < 4; ++j)
        mma_ts_warp(tmem + kTO, tmem + kTP + 8u * j, sdesc_mn(vt + 2048u * j), id_o, (first && j == 0) ? 0u : 1u);
      mma_commit_warp(barx(G::kODone));
      mma_commit_warp(barx(G::kVFree + (k & 1)));
    };
    // event-driven: S(k) once its K operands are in (both sides), S(k - 1) was read and, for an
    // item's first tile, its queries are in; O(k) once its V' and P(k) are in.  Nothing ready:
    // a short sleep, so that the poll does not take issue slots from the SMSP's other warps.
    int ns = 0, no = 0, end = 1 << 30, items = 0;
    uint32_t firsts = 0u;                              // bit k % 32: tile k opens its item
    long long idle = 0;
    while (no < end) {
      bool did = false;
      if (ns < end && ns <= no + 2 && uni(bar_poll(barx(G::kKOps + (ns & 1)), (ns >> 1) & 1))) {
        const CDesc dn = desc[ns & 3];
        const bool fin = uni(dn.item < 0), first = uni(dn.first != 0);
        if (fin) {
          end = ns;
          did = true;
        } else if ((ns == 0 || uni(bar_poll(barx(G::kSEmpty), (ns - 1) & 1))) &&
                   (!first || uni(bar_poll(barx(G::kQReady), items & 1)))) {
          items += first ? 1 : 0;
          issue_s(ns);
          firsts = first ? (firsts | (1u << (ns & 31))) : (firsts & ~(1u << (ns & 31)));
          ++ns;
          did = true;
        }
      }
      if (no < ns && uni(bar_poll(barx(G::kVOps + (no & 1)), (no >> 1) & 1)) && uni(bar_poll(barx(G::kPFull), no & 1))) {
        issue_o(no, (firsts >> (no & 31)) & 1u);
        ++no;
        did = true;
      }
      if (did) {
        idle = 0;
      } else {
        if (++idle > kCPollLimit) {
          failed = true;
          break;
        }
        __nanosleep(32);
      }
    }
    mma_commit_warp(barx(G::kDrain));                  // every MMA issued completes before the CTA ends
    bool f2 = false;
    (void)bar_wait(barx(G::kDrain), 0, f2);
    __syncwarp();
  } else if (warp < 8 || warp >= 16) {
    // ---- operands: K side on warps 4, 5, 16, 17 (the first two SMSPs): K^ rows and the
    // token factors; V side on warps 2, 3, 6, 7 (the other two): the sign rows A', then
    // V' and the ones column.  A tile's S MMAs wait for both sides' K-operand arrivals;
    // the V side builds A'(k) as soon as S(k - 2) has run, ahead of V'(k) --------------------
    const bool vside = warp < 4 || (warp >= 6 && warp < 8);
    const int ridx = vside ? (warp < 4 ? warp - 2 : warp - 4) : (warp < 8 ? warp - 4 : warp - 14);
    const int u = 32 * ridx + lane + (vside ? 128 : 0);   // K side 0 .. 127, V side 128 .. 255
    const int t = u & 63, hf = (u >> 6) & 1;           // token row, channel (projection) half (warp-uniform)
    const uint32_t lane_off = static_cast<uint32_t>(lane) * 4u;
    for (int seq = 0;; ++seq) {
      const int s = seq % kCStages, buf = seq & 1;
      bool ok = bar_wait(barx(G::kRecFull + s), (seq / kCStages) & 1, failed);
      if (seq >= 2)                                    // the S MMAs of two tiles back have read K^ and A'
        ok = bar_wait(barx(G::kKFree + buf), ((seq - 2) >> 1) & 1, failed) && ok;
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      const CDesc d = rec_desc[s];
      const uint32_t rec = sb + G::REC + s * G::STAGE;
      const uint32_t ob = sb + G::OPS + buf * G::OPS_BYTES;
      const int pg = t >> 4, slot = t & 15;
      const bool tv = d.item >= 0 && t < d.npos && ((d.mask >> pg) & 1u);
      const uint32_t kb = rec + pg * G::PAGE;
      if (!vside) {
        if (d.item >= 0) {
          float fa = 0.0f;
          if (tv)
            fa = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(kb + G::K_NORM + 2 * slot)))) *
                 kInvSqrtDC;
          if (hf == 0)
            half_rows<KBH, false>(ob + G::KH, kb + slot * G::CBK, t, 0, tv, sb + G::LUT + lut_off(KBH) + lane_off, __half2());
          else
            half_rows<KBL, false>(ob + G::KH, kb + slot * G::CBK + 8 * KBH, t, 1, tv, sb + G::LUT + lut_off(KBL) + lane_off,
                                  __half2());
          if (hf == 0) {
            const uint32_t fac = sb + G::FAC + (seq & 3) * 512;
            stsf(fac + 4 * t, fa * a.scale_log2);
            stsf(fac + 256 + 4 * t, tv ? 0.0f : -INFINITY);
          }
        }
        if (u == 0) desc[seq & 3] = d;
        fence_async_smem();                             // the operand tiles, for the tensor cores
        __syncwarp();
        if (lane == 0) {
          bar_arrive(barx(G::kKOps + buf));
          bar_arrive(barx(G::kDescFull + (seq & 3)));
          if (d.item >= 0) bar_arrive(barx(G::kRecEmpty + s));
        }
        if (d.item < 0) break;
        continue;
      }
      // V side: A' = (fb / fa)(2 b - 1) for the 64 projections of this half (zero for a missing token)
      if (QJL && d.item >= 0) {
        float ratio = 0.0f;
        uint2 sw = make_uint2(0u, 0u);
        if (tv) {
          const float nk = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(kb + G::K_NORM + 2 * slot))));
          const float rk = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(kb + G::K_RNORM + 2 * slot))));
          sw = lds64(kb + G::K_SIGNS + slot * 16 + 8 * hf);
          const float fa = nk * kInvSqrtDC, fb = rk * (kSqrtHalfPiC / 128.0f);
          ratio = fa > 0.0f ? fb / fa : 0.0f;
        }
        const __half2 fb2 = __float2half2_rn(ratio);
        const uint32_t fbv = tv ? *reinterpret_cast<const uint32_t*>(&fb2) : 0u;   // |A'| in both halves
        const uint32_t vm = tv ? 0xFFFFFFFFu : 0u;
        const uint32_t st = sb + G::SGN + lane_off * 2;
#pragma unroll 1
        for (int cc = 0; cc < 8; cc += 2) {               // two chunks per step, loads first
          const uint32_t w = cc < 4 ? sw.x : sw.y;
          const uint32_t b0 = __byte_perm(w, 0u, 0x4440u + (cc & 3)), b1 = __byte_perm(w, 0u, 0x4441u + (cc & 3));
          const uint2 l0 = lds64(st + (b0 & 0xFu) * 256u), h0 = lds64(st + (b0 >> 4) * 256u);
          const uint2 l1 = lds64(st + (b1 & 0xFu) * 256u), h1 = lds64(st + (b1 >> 4) * 256u);
          sts128(ob + G::AS + chunk_off(t, 8 * hf + cc, kCT), fbv | (l0.x & vm), fbv | (l0.y & vm), fbv | (h0.x & vm),
                 fbv | (h0.y & vm));
          sts128(ob + G::AS + chunk_off(t, 8 * hf + cc + 1, kCT), fbv | (l1.x & vm), fbv | (l1.y & vm),
                 fbv | (h1.x & vm), fbv | (h1.y & vm));
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) bar_arrive(barx(G::kKOps + buf));
      if (d.item < 0) break;
      // V' rows, once the O MMAs of two tiles back have read the buffer
      ok = seq < 2 || bar_wait(barx(G::kVFree + buf), ((seq - 2) >> 1) & 1, failed);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      {
        const uint32_t vb = kb + G::KBB;
        float fv = 0.0f;
        if (tv)
          fv = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(vb + G::V_NORM + 2 * slot)))) * kInvSqrtDC;
        const __half2 fv2 = __float2half2_rn(fv);
        if (hf == 0) {
          half_rows<VBH, true>(ob + G::VT, vb + slot * G::CBV, t, 0, tv, sb + G::LUT + lut_off(VBH) + lane_off, fv2);
          // channels 128 .. 143: 1 in channel 128 for a token that is there, else 0
          sts128(ob + G::VT + chunk_off(t, 16, kCT), tv ? 0x3C00u : 0u, 0u, 0u, 0u);
          sts128(ob + G::VT + chunk_off(t, 17, kCT), 0u, 0u, 0u, 0u);
        } else {
          half_rows<VBL, true>(ob + G::VT, vb + slot * G::CBV + 8 * VBH, t, 1, tv, sb + G::LUT + lut_off(VBL) + lane_off,
                               fv2);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        bar_arrive(barx(G::kVOps + buf));
        bar_arrive(barx(G::kRecEmpty + s));
      }
    }
  } else {
    // ---- softmax (thread = query row of the item, tensor-memory lane r) --------------------
    const int e = warp - 8;                            // 0 .. 7
    const int wq = warp & 3, hh = e >> 2, r = 32 * wq + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * wq) << 16);
    float m_run = kNegBigC;
    int row_end = 0;                                   // exclusive causal end of this row
    long long blk = 0;                                 // the item's query block (b H + h) nqb + qb
    int chunk = 0, wmin_end = 0;
    for (int seq = 0;; ++seq) {
      bool ok = bar_wait(barx(G::kDescFull + (seq & 3)), (seq >> 2) & 1, failed);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      const CDesc d = desc[seq & 3];
      if (d.item < 0) break;
      if (d.first) {
        chunk = d.chunk;
        const int rr = kCR * d.qb + r;                 // row t G + g among the sequence's new tokens
        row_end = rr < rows_all ? d.start + rr / a.G + 1 : 0;
        int me = rr < rows_all ? row_end : 0x7FFFFFFF;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) me = min(me, __shfl_xor_sync(0xffffffffu, me, o));
        wmin_end = me;
        // this row's q~ hi/lo and u words (written by the query prep in column order), half
        // hh of each: columns 32 hh .. 32 hh + 31 of the three blocks
        blk = (static_cast<long long>(d.b) * a.H + d.h) * nqb + d.qb;
        const uint4* src = rr < rows_all ? reinterpret_cast<const uint4*>(a.qprep) + blk * 48 * 128 + r : nullptr;
        {
          uint4 x[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            x[i] = src ? src[(8 * hh + i) * 128] : make_uint4(0u, 0u, 0u, 0u);
            x[8 + i] = src ? src[(16 + 8 * hh + i) * 128] : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int bk = 0; bk < 2; ++bk)
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
              uint32_t w[16];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 v = x[8 * bk + 4 * h16 + i];
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
              }
              tst16(trow + (bk ? kTQL : kTQH) + 32u * hh + 16u * h16, w);
            }
        }
        if (QJL) {
          uint4 x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = src ? src[(32 + 8 * hh + i) * 128] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int h16 = 0; h16 < 2; ++h16) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 v = x[4 * h16 + i];
              w[4 * i] = v.x;
              w[4 * i + 1] = v.y;
              w[4 * i + 2] = v.z;
              w[4 * i + 3] = v.w;
            }
            tst16(trow + kTU + 32u * hh + 16u * h16, w);
          }
        }
        tst_wait();
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(barx(G::kQReady));
        m_run = kNegBigC;
      }
      // this tile's scores (tokens 32 hh .. 32 hh + 31): read, release, logits
      ok = bar_wait(barx(G::kSFull), seq & 1, failed);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
      tc_after();
      float x[32];
      tld32(trow + kTS + 32u * hh, x);
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(barx(G::kSEmpty));
      {
        const uint32_t fac = sb + G::FAC + (seq & 3) * 512 + 128u * hh;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const uint4 fa = lds128(fac + 16 * j4), bi = lds128(fac + 256 + 16 * j4);
          x[4 * j4] = fmaf(__uint_as_float(fa.x), x[4 * j4], __uint_as_float(bi.x));
          x[4 * j4 + 1] = fmaf(__uint_as_float(fa.y), x[4 * j4 + 1], __uint_as_float(bi.y));
          x[4 * j4 + 2] = fmaf(__uint_as_float(fa.z), x[4 * j4 + 2], __uint_as_float(bi.z));
          x[4 * j4 + 3] = fmaf(__uint_as_float(fa.w), x[4 * j4 + 3], __uint_as_float(bi.w));
        }
      }
      const int pbase = d.p0 + 32 * hh;
      if (pbase + 32 > wmin_end) {                     // the causal end falls inside (or before) these tokens
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = pbase + j < row_end ? x[j] : -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) mx = fmaxf(mx, x[j]);
      // the pair's row max: through shared memory, double-buffered by tile parity
      {
        float* xm = reinterpret_cast<float*>(sm + G::XMAX) + (seq & 1) * 256;
        xm[hh * 128 + r] = mx;
        __syncwarp();
        if (lane == 0) bar_arrive(barx(G::kXch + 2 * wq + (seq & 1)));
        ok = bar_wait(barx(G::kXch + 2 * wq + (seq & 1)), (seq >> 1) & 1, failed);
        if (!__all_sync(0xffffffffu, ok)) {
          failed = true;
          break;
        }
        mx = fmaxf(mx, xm[(1 - hh) * 128 + r]);
      }
      // the previous tile's O MMA has read P and updated O before either changes
      if (!d.first) {
        ok = bar_wait(barx(G::kODone), (seq - 1) & 1, failed);
        if (!__all_sync(0xffffffffu, ok)) {
          failed = true;
          break;
        }
        tc_after();
      }
      const bool moved = mx > m_run + kLazyC;         // the running max moves: rescale this row of O and l
      float alpha = 1.0f;
      if (moved) {
        alpha = exp2f(m_run - mx);
        m_run = mx;
      }
      if (!d.first && __any_sync(0xffffffffu, moved)) {   // warp-wide: the tensor-memory accesses are collective
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          float o[16];
          uint32_t ou[16];
          const uint32_t col = kTO + 64u * hh + 16u * q4;
          tld16(trow + col, o);
#pragma unroll
          for (int k = 0; k < 16; ++k) ou[k] = __float_as_uint(o[k] * alpha);
          tst16(trow + col, ou);
        }
        if (hh == 0) tst1(trow + kTO + 128u, __float_as_uint(__uint_as_float(tld1(trow + kTO + 128u)) * alpha));
        tst_wait();
      }
      uint32_t pp[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const __half2 h2 = __floats2half2_rn(ex2_ftz(x[2 * k] - m_run), ex2_ftz(x[2 * k + 1] - m_run));
        pp[k] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      tst16(trow + kTP + 16u * hh, pp);
      tst_wait();
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(barx(G::kPFull));
      if (d.last) {                                    // the item's partial (max, sum, O) for this row
        ok = bar_wait(barx(G::kODone), seq & 1, failed);
        if (!__all_sync(0xffffffffu, ok)) {
          failed = true;
          break;
        }
        tc_after();
        // stored by query block, row-minor: a warp's stores are 128 contiguous bytes
        float* dst = a.part + ((blk * nch + chunk) * (kD + 2)) * 128 + r;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          float o[16];
          tld16(trow + kTO + 64u * hh + 16u * q4, o);
#pragma unroll
          for (int k = 0; k < 16; ++k) dst[(2 + 64 * hh + 16 * q4 + k) * 128] = o[k];
        }
        if (hh == 0) {
          const float l = __uint_as_float(tld1(trow + kTO + 128u));
          dst[0] = m_run;
          dst[128] = l;
        }
        tc_before();
      }
    }
  }
  if (failed) atomicOr(a.tab.err, kErrTimeout);
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

template <int A, int B, int C, int D, typename F>
bool launch_widths(std::integer_sequence<int, A, B, C, D>, F&& f) {
  return f(std::integral_constant<int, A>{}, std::integral_constant<int, B>{}, std::integral_constant<int, C>{},
           std::integral_constant<int, D>{});
}

template <int KBH, int KBL, int VBH, int VBL, bool QJL>
bool layout_matches(const KindLayout& kl, const KindLayout& vl) {
  using G = CGeo<KBH, KBL, VBH, VBL, QJL>;
  return kl.block_bytes == G::KBB && vl.block_bytes == G::VBB && kl.code_bytes == G::CBK && vl.code_bytes == G::CBV &&
         kl.off_norm == G::K_NORM && (!QJL || (kl.off_signs == G::K_SIGNS && kl.off_rnorm == G::K_RNORM)) &&
         vl.off_norm == G::V_NORM;
}

template <int KBH, int KBL, int VBH, int VBL, bool QJL>
cudaError_t launch_causal_tc_t(const DecodeArgs& a, int items, int nqb, int grid, cudaStream_t s) {
  using G = CGeo<KBH, KBL, VBH, VBL, QJL>;
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e = smem_attr_once(causal_tc_kernel<KBH, KBL, VBH, VBL, QJL>, G::SMEM, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(causal_tc_kernel<KBH, KBL, VBH, VBL, QJL>, dim3(grid), dim3(kCThreadsTC),
                    static_cast<size_t>(G::SMEM), s, a, items, nqb);
}

// The bit widths (K high, K low, V high, V low) with a compiled instance.
template <typename F>
bool with_widths(const KindLayout& kl, const KindLayout& vl, F&& f) {
  switch (kl.g[0].bits * 1000 + kl.g[1].bits * 100 + vl.g[0].bits * 10 + vl.g[1].bits) {
    case 3333: return f(std::integer_sequence<int, 3, 3, 3, 3>{});
    case 4343: return f(std::integer_sequence<int, 4, 3, 4, 3>{});
    case 3232: return f(std::integer_sequence<int, 3, 2, 3, 2>{});
    case 4444: return f(std::integer_sequence<int, 4, 4, 4, 4>{});
    case 2222: return f(std::integer_sequence<int, 2, 2, 2, 2>{});
    case 4422: return f(std::integer_sequence<int, 4, 4, 2, 2>{});
    default: return false;
  }
}

}  // namespace

int causal_tc_block_rows() { return kCR; }
int causal_tc_max_chunk() { return kCMaxChunk; }

bool causal_tc_supported(const KindLayout& kl, const KindLayout& vl, int m) {
  if (m != 128 || kl.split != 64 || vl.split != 64) return false;
  // one lookup table per bit width: every group of that width has the same centroids
  const GroupBook* gs[4] = {&kl.g[0], &kl.g[1], &vl.g[0], &vl.g[1]};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (gs[i]->bits == gs[j]->bits)
        for (int k = 0; k < (1 << gs[i]->bits); ++k)
          if (gs[i]->c[k] != gs[j]->c[k]) return false;
  return with_widths(kl, vl, [&](auto w) {
    return launch_widths(w, [&](auto kbh, auto kbl, auto vbh, auto vbl) {
      constexpr int KH = decltype(kbh)::value, KL = decltype(kbl)::value, VH = decltype(vbh)::value,
                    VL = decltype(vbl)::value;
      return kl.qjl ? layout_matches<KH, KL, VH, VL, true>(kl, vl) : layout_matches<KH, KL, VH, VL, false>(kl, vl);
    });
  });
}

cudaError_t launch_causal_tc(const DecodeArgs& a, int nqb, cudaStream_t s) {
  const long long items = static_cast<long long>(a.B) * a.H * nqb * a.nchunks;
  if (items < 1 || items > (1LL << 30) || a.chunk < kPage || a.chunk > kCMaxChunk || a.chunk % kPage)
    return cudaErrorInvalidValue;
  int dev = 0, sms = 152;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(items < sms ? items : sms);
  const int n = static_cast<int>(items);
  e = cudaErrorInvalidValue;
  with_widths(a.kl, a.vl, [&](auto w) {
    return launch_widths(w, [&](auto kbh, auto kbl, auto vbh, auto vbl) {
      constexpr int KH = decltype(kbh)::value, KL = decltype(kbl)::value, VH = decltype(vbh)::value,
                    VL = decltype(vbl)::value;
      e = a.kl.qjl ? launch_causal_tc_t<KH, KL, VH, VL, true>(a, n, nqb, grid, s)
                   : launch_causal_tc_t<KH, KL, VH, VL, false>(a, n, nqb, grid, s);
      return true;
    });
  });
  return e;
}

}  // namespace tq
