// Decode attention, split-K partials stage, on the tensor cores.
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.2 (decode: one query per
// head against every cached key, softmax, weighted sum of values), §4.2 (the
// codebook is only looked up at run time), §4.3 (stage-1 score plus the 1-bit
// QJL correction; softmax(QK^T/sqrt(d))); [P2] "생각정리 209 (TurboQuant)", stage 2.
//
// Per CTA: one (chunk, KV head, sequence); 4 warps, each owns whole 16-token
// pages of the chunk and keeps its own online-softmax state.  Per page:
//   * the packed K and V blocks of the page are staged into shared memory by
//     two bulk copies (cp.async.bulk, mbarrier completion, 3-stage ring/warp);
//   * codes are turned into fp16 directly inside mma.sync fragments: a
//     prmt byte-table lookup per 4 codes reads the low and high bytes of the
//     fp16 centroids (no shared-memory lookup table); QJL sign bits become
//     +-1.0 halves with one shift + lop3 per pair;
//   * scores: S1 = K^ Q~^T and S2 = sign * U^T, m16n8k16 with the 16 tokens on
//     M and the G <= 8 query heads of the KV head on N (K = channels);
//   * logits = (n_k/sqrt(d) S1 + sqrt(pi/2)/m rho S2) * scale; online softmax
//     on the accumulator fragments (max over 8 lanes by 3 shuffles);
//   * P' = p * n_v / sqrt(d) goes through a 256-byte shared tile to become the
//     B operand of O^T += V^^T P'^T (M = channels, 8 tiles; K = tokens); the
//     V^ fragments pair one channel of two tokens, built by re-pairing the
//     per-token lookups with one prmt per half2.
// The channel order inside the fragments is a fixed permutation chosen so that
// every thread reads contiguous code bits; Q~, U and the output use the same
// permutation, so the contraction is unchanged.
//
// Supported here: d = 128, m = 128, channel split 64, 2-4 bits per group.
// Other configurations run the CUDA-core kernel in tq_decode.cu.

#include "tq_internal.h"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 3;
constexpr float kInvSqrtD = 0.08838834764831845f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;
constexpr int kWaitLimit = 1 << 22;
// Finite "minus infinity": exp2 of (sentinel - finite) is exactly 0, and an
// all-empty chunk ends with max = sentinel, acc = 0, so its merge weight or
// its value is 0 either way; no -inf tests are needed around exp2.
constexpr float kNegBig = -1.0e30f;

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for phase `parity` of an mbarrier; false after kWaitLimit polls.
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
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// fp16 codebook tables held in registers, one per channel group
// ---------------------------------------------------------------------------
struct Tab {
  uint32_t l0, l1, h0, h1;   // low / high bytes of 8 fp16 values (b = 2 uses l0 = low, l1 = high)
};

__device__ __forceinline__ uint32_t f16bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

// b = 3: the 8 centroids; b = 4: the 8 positive centroids (magnitudes); b = 2: 4 centroids.
template <int B>
__device__ Tab make_tab(const float* c) {
  Tab t{0u, 0u, 0u, 0u};
  if (B == 2) {
    for (int k = 0; k < 4; ++k) {
      uint32_t h = f16bits(c[k]);
      t.l0 |= (h & 0xFFu) << (8 * k);
      t.l1 |= (h >> 8) << (8 * k);
    }
  } else {
    const int base = (B == 4) ? 8 : 0;
    for (int k = 0; k < 8; ++k) {
      uint32_t h = f16bits(c[base + k]);
      uint32_t lo = h & 0xFFu, hi = h >> 8;
      if (k < 4) {
        t.l0 |= lo << (8 * k);
        t.h0 |= hi << (8 * k);
      } else {
        t.l1 |= lo << (8 * (k - 4));
        t.h1 |= hi << (8 * (k - 4));
      }
    }
  }
  return t;
}

// Pairing of the 8 channels of a chunk inside the 4 half2 a lookup produces:
// half2 j holds (chunk channel PLO[j] in the low half, PHI[j] in the high half).
__host__ __device__ constexpr int pair_lo(int B, int j) {
  return B == 2 ? (j == 0 ? 0 : j == 1 ? 4 : j == 2 ? 1 : 5) : B == 3 ? 2 * j : j;
}
__host__ __device__ constexpr int pair_hi(int B, int j) {
  return B == 2 ? (j == 0 ? 2 : j == 1 ? 6 : j == 2 ? 3 : 7) : B == 3 ? 2 * j + 1 : j + 4;
}

// 8 consecutive codes of one vector (8*B bits in the low bits of v) -> 4 half2.
template <int B>
__device__ __forceinline__ void deq8(uint32_t v, const Tab& t, uint32_t (&h)[4]);

template <>
__device__ __forceinline__ void deq8<3>(uint32_t v, const Tab& t, uint32_t (&h)[4]) {
  // stored octet: channels 0-5 already in nibbles; channels 6, 7 in the spare
  // bit 3 of each nibble, gathered into nibbles 6, 7 by one multiply
  // (bits 3/11/19 -> 24/25/26, 7/15/23 -> 28/29/30; the other partial
  // products land on distinct bits below 24, so nothing carries)
  const uint32_t xm = v & 0x00777777u;
  const uint32_t sp = (v & 0x00888888u) * 0x00204080u;
  const uint32_t x = xm | (sp & 0x77000000u);
  const uint32_t xh = x >> 16;
  const uint32_t rl0 = prmt(t.l0, t.l1, x), rh0 = prmt(t.h0, t.h1, x);
  const uint32_t rl1 = prmt(t.l0, t.l1, xh), rh1 = prmt(t.h0, t.h1, xh);
  h[0] = prmt(rl0, rh0, 0x5140u);
  h[1] = prmt(rl0, rh0, 0x7362u);
  h[2] = prmt(rl1, rh1, 0x5140u);
  h[3] = prmt(rl1, rh1, 0x7362u);
}

template <>
__device__ __forceinline__ void deq8<4>(uint32_t w, const Tab& t, uint32_t (&h)[4]) {
  // stored sign-magnitude nibbles: bit 3 = negative half, bits 0-2 = rank of |centroid|
  const uint32_t neg = w & 0x88888888u;
  const uint32_t idx = w & 0x77777777u;
  const uint32_t a = prmt(idx, 0u, 0x0020u);                   // nibbles n0 n1 n4 n5
  const uint32_t b = prmt(idx, 0u, 0x0031u);                   // nibbles n2 n3 n6 n7
  const uint32_t rla = prmt(t.l0, t.l1, a), rha = prmt(t.h0, t.h1, a);
  const uint32_t rlb = prmt(t.l0, t.l1, b), rhb = prmt(t.h0, t.h1, b);
  h[0] = prmt(rla, rha, 0x6240u) | ((neg << 12) & 0x80008000u);   // (n0, n4)
  h[1] = prmt(rla, rha, 0x7351u) | ((neg << 8) & 0x80008000u);    // (n1, n5)
  h[2] = prmt(rlb, rhb, 0x6240u) | ((neg << 4) & 0x80008000u);    // (n2, n6)
  h[3] = prmt(rlb, rhb, 0x7351u) | (neg & 0x80008000u);           // (n3, n7)
}

template <>
__device__ __forceinline__ void deq8<2>(uint32_t v, const Tab& t, uint32_t (&h)[4]) {
  const uint32_t x = v & 0x3333u;           // c0 c2 c4 c6
  const uint32_t y = (v >> 2) & 0x3333u;    // c1 c3 c5 c7
  const uint32_t rlx = prmt(t.l0, t.l1, x), rhx = prmt(t.l0, t.l1, x | 0x4444u);
  const uint32_t rly = prmt(t.l0, t.l1, y), rhy = prmt(t.l0, t.l1, y | 0x4444u);
  h[0] = prmt(rlx, rhx, 0x5140u);   // (c0, c2)
  h[1] = prmt(rlx, rhx, 0x7362u);   // (c4, c6)
  h[2] = prmt(rly, rhy, 0x5140u);   // (c1, c3)
  h[3] = prmt(rly, rhy, 0x7362u);   // (c5, c7)
}

// The 8*B-bit field at bit offset `off` of a word array in shared memory
// (4-bit fields are word aligned and need no shift).
template <int B>
__device__ __forceinline__ uint32_t field(const uint32_t* row, int off) {
  if (B == 4) return row[off >> 5];
  const int w = off >> 5, sh = off & 31;
  return __funnelshift_r(row[w], row[w + 1], sh);
}

// QJL sign pair (projections k, k+16 of a 32-bit word): +1.0 if the bit is set, else -1.0.
__device__ __forceinline__ uint32_t sign_pair(uint32_t notw, int k) {
  return ((notw << (15 - k)) & 0x80008000u) | 0x3C003C00u;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return static_cast<uint32_t>(f16bits(lo)) | (static_cast<uint32_t>(f16bits(hi)) << 16);
}

// Physical channel of the low/high half of pair p (0..15) of thread t on the K side.
template <int KBH, int KBL>
__device__ __forceinline__ void k_pair_channels(int t, int p, int& clo, int& chi) {
  const int u = p >> 2, j = p & 3;
  const int b = u < 2 ? KBH : KBL;
  const int base = 32 * u + 8 * t;
  clo = base + pair_lo(b, j);
  chi = base + pair_hi(b, j);
}

template <int B>
__device__ __forceinline__ int pair_of_channel(int c, bool& high) {
  for (int j = 0; j < 4; ++j) {
    if (pair_lo(B, j) == c) { high = false; return j; }
    if (pair_hi(B, j) == c) { high = true; return j; }
  }
  high = false;
  return 0;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int KBH, int KBL, int VBH, int VBL, bool QJL>
__global__ void __launch_bounds__(kThreads, 3) chunk_mma_kernel(DecodeArgs a) {
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  constexpr int CBK = (64 * KBH + 64 * KBL) / 8;     // code bytes per key
  constexpr int CBV = (64 * VBH + 64 * VBL) / 8;
  constexpr int KBB = 16 * (CBK + (QJL ? 16 + 2 : 0) + 2);   // K block bytes (m = 128)
  constexpr int VBB = 16 * (CBV + 2);
  constexpr int STAGE = KBB + VBB;
  constexpr int K_SIGNS = 16 * CBK;
  constexpr int K_NORM = K_SIGNS + (QJL ? 16 * 16 : 0);
  constexpr int K_RNORM = K_NORM + 32;
  constexpr int V_NORM = 16 * CBV;

  __shared__ __align__(128) unsigned char stage_buf[kWarps][kStages][STAGE];
  __shared__ __align__(8) unsigned long long bars[kWarps][kStages];
  __shared__ int stage_valid[kWarps][kStages];
  __shared__ __align__(16) __half ptile[kWarps][8][16];
  __shared__ float red_m[kWarps][8];
  __shared__ float red_l[kWarps][8];
  __shared__ float red_acc[kWarps][8][kD];

  // ---- per-thread constants: tables and query fragments --------------------
  const Tab tk0 = make_tab<KBH>(a.kl.g[0].c), tk1 = make_tab<KBL>(a.kl.g[1].c);
  const Tab tv0 = make_tab<VBH>(a.vl.g[0].c), tv1 = make_tab<VBL>(a.vl.g[1].c);

  const bool head_ok = g < a.G;
  const float* qrow = a.qprep + (static_cast<long long>(b) * a.Hq + h * a.G + (head_ok ? g : 0)) * (kD + a.m);
  uint32_t qf[16], uf[16];
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    int clo, chi;
    k_pair_channels<KBH, KBL>(t, p, clo, chi);
    qf[p] = head_ok ? pack_h2(qrow[clo], qrow[chi]) : 0u;
    const int plo = 32 * t + (p), phi = plo + 16;          // sign pair p of word t: projections (p, p+16)
    uf[p] = (QJL && head_ok) ? pack_h2(qrow[kD + plo], qrow[kD + phi]) : 0u;
  }

  int L = a.seq_lens[b] + a.len_add;
  if (L < 0 || L > a.max_seq_len || L > a.maxp * kPage) {
    if (threadIdx.x == 0 && chunk == 0 && h == 0) atomicOr(a.tab.err, kErrSeqLen);
    L = L < 0 ? 0 : L;
    L = L > a.max_seq_len ? a.max_seq_len : L;
    L = L > a.maxp * kPage ? a.maxp * kPage : L;
  }
  const int t0 = chunk * a.chunk;
  const int t1 = min(t0 + a.chunk, L);
  const int npages = t1 > t0 ? (t1 - t0 + kPage - 1) / kPage : 0;
  const int p0 = t0 / kPage;
  const int* bt_row = a.block_table + static_cast<long long>(b) * a.maxp;
  const unsigned char* kbase = a.kc + static_cast<long long>(h) * KBB;
  const unsigned char* vbase = a.vc + static_cast<long long>(h) * VBB;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  auto issue = [&](int i) {       // lane 0: stage the i-th page of this warp
    const int k = warp + kWarps * i;
    const int s = i % kStages;
    const uint32_t bar = smem_u32(&bars[warp][s]);
    const int page = bt_row[p0 + k];
    if (page < 0 || page >= a.num_pages) {
      atomicOr(a.tab.err, kErrPage);
      stage_valid[warp][s] = 0;
      mbar_arrive(bar);
      return;
    }
    stage_valid[warp][s] = 1;
    fence_proxy_async();
    mbar_arrive_tx(bar, STAGE);
    bulk_g2s(smem_u32(&stage_buf[warp][s][0]), kbase + static_cast<long long>(page) * a.k_page_bytes, KBB, bar);
    bulk_g2s(smem_u32(&stage_buf[warp][s][KBB]), vbase + static_cast<long long>(page) * a.v_page_bytes, VBB, bar);
  };

  const int my_pages = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;
  if (lane == 0) {
    for (int i = 0; i < kStages && i < my_pages; ++i) issue(i);
  }
  __syncwarp();

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  float m_run[2] = {kNegBig, kNegBig};
  float l_run[2] = {0.0f, 0.0f};
  const float k1 = kInvSqrtD * a.scale_log2;
  const float k2 = kSqrtHalfPi / 128.0f * a.scale_log2;
  bool failed = false;

  for (int i = 0; i < my_pages; ++i) {
    const int s = i % kStages;
    if (!failed && !mbar_wait(smem_u32(&bars[warp][s]), (i / kStages) & 1)) {
      failed = true;
      if (lane == 0) atomicOr(a.tab.err, kErrTimeout);
    }
    const int k = warp + kWarps * i;
    const int pbase = (p0 + k) * kPage;
    const bool pvalid = !failed && stage_valid[warp][s];
    const unsigned char* kb = &stage_buf[warp][s][0];
    const unsigned char* vb = &stage_buf[warp][s][KBB];

    // ---- scores ---------------------------------------------------------
    float s1[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t* rg = reinterpret_cast<const uint32_t*>(kb + g * CBK);
      const uint32_t* rg8 = reinterpret_cast<const uint32_t*>(kb + (g + 8) * CBK);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t ha[4], hb[4];
        if (u < 2) {
          const int off = 32 * u * KBH + 8 * t * KBH;
          deq8<KBH>(field<KBH>(rg, off), tk0, ha);
          deq8<KBH>(field<KBH>(rg8, off), tk0, hb);
        } else {
          const int off = 64 * KBH + 32 * (u - 2) * KBL + 8 * t * KBL;
          deq8<KBL>(field<KBL>(rg, off), tk1, ha);
          deq8<KBL>(field<KBL>(rg8, off), tk1, hb);
        }
        mma16816(s1, ha[0], hb[0], ha[1], hb[1], qf[4 * u + 0], qf[4 * u + 1]);
        mma16816(s1, ha[2], hb[2], ha[3], hb[3], qf[4 * u + 2], qf[4 * u + 3]);
      }
      if (QJL) {
        const uint32_t* sg = reinterpret_cast<const uint32_t*>(kb + K_SIGNS);
        const uint32_t na = ~sg[g * 4 + t], nb = ~sg[(g + 8) * 4 + t];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          mma16816(s2, sign_pair(na, 2 * st), sign_pair(nb, 2 * st), sign_pair(na, 2 * st + 1),
                   sign_pair(nb, 2 * st + 1), uf[2 * st], uf[2 * st + 1]);
        }
      }
    }
    const __half* nk = reinterpret_cast<const __half*>(kb + K_NORM);
    const __half* rk = reinterpret_cast<const __half*>(kb + K_RNORM);
    const __half* nv = reinterpret_cast<const __half*>(vb + V_NORM);
    const bool vg = pvalid && pbase + g < t1;
    const bool vg8 = pvalid && pbase + g + 8 < t1;
    float lg[4];
    {
      const float nkg = __half2float(nk[g]), nkg8 = __half2float(nk[g + 8]);
      const float rkg = QJL ? __half2float(rk[g]) : 0.f, rkg8 = QJL ? __half2float(rk[g + 8]) : 0.f;
      lg[0] = vg ? fmaf(nkg * k1, s1[0], rkg * k2 * s2[0]) : kNegBig;
      lg[1] = vg ? fmaf(nkg * k1, s1[1], rkg * k2 * s2[1]) : kNegBig;
      lg[2] = vg8 ? fmaf(nkg8 * k1, s1[2], rkg8 * k2 * s2[2]) : kNegBig;
      lg[3] = vg8 ? fmaf(nkg8 * k1, s1[3], rkg8 * k2 * s2[3]) : kNegBig;
    }
    // ---- online softmax over this page (heads 2t, 2t+1) -------------------
    float pr[4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float mx = fmaxf(lg[c], lg[c + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[c], mx);
      const float alpha = exp2f(m_run[c] - m_new);
      pr[c] = exp2f(lg[c] - m_new);
      pr[c + 2] = exp2f(lg[c + 2] - m_new);
      l_run[c] = fmaf(l_run[c], alpha, pr[c] + pr[c + 2]);
      m_run[c] = m_new;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][c] *= alpha;
        acc[mt][c + 2] *= alpha;
      }
    }
    // ---- P' = p * nv / sqrt(d) into the transposed shared tile -------------
    {
      const float wg = vg ? __half2float(nv[g]) * kInvSqrtD : 0.0f;
      const float wg8 = vg8 ? __half2float(nv[g + 8]) * kInvSqrtD : 0.0f;
      ptile[warp][2 * t][g] = __float2half_rn(pr[0] * wg);
      ptile[warp][2 * t + 1][g] = __float2half_rn(pr[1] * wg);
      ptile[warp][2 * t][g + 8] = __float2half_rn(pr[2] * wg8);
      ptile[warp][2 * t + 1][g + 8] = __float2half_rn(pr[3] * wg8);
    }
    __syncwarp();
    const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(&ptile[warp][g][2 * t]);
    const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(&ptile[warp][g][2 * t + 8]);
    // ---- O^T += V^^T P'^T ---------------------------------------------------
    {
      uint32_t fa[8][2], fb[8][2];   // [m-tile][token pair]: chunk A (rows g), chunk B (rows g+8)
#pragma unroll
      for (int tp = 0; tp < 2; ++tp) {
        const int ta = 2 * t + 8 * tp;   // tokens ta, ta+1
        const uint32_t* r0 = reinterpret_cast<const uint32_t*>(vb + ta * CBV);
        const uint32_t* r1 = reinterpret_cast<const uint32_t*>(vb + (ta + 1) * CBV);
        uint32_t x0[4], x1[4];
        // chunk A: channels 8g..8g+7 (hi group)
        deq8<VBH>(field<VBH>(r0, 8 * g * VBH), tv0, x0);
        deq8<VBH>(field<VBH>(r1, 8 * g * VBH), tv0, x1);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          bool hi;
          const int j = pair_of_channel<VBH>(c, hi);
          fa[c][tp] = prmt(x0[j], x1[j], hi ? 0x7632u : 0x5410u);
        }
        // chunk B: channels 64+8g..64+8g+7 (lo group)
        deq8<VBL>(field<VBL>(r0, 64 * VBH + 8 * g * VBL), tv1, x0);
        deq8<VBL>(field<VBL>(r1, 64 * VBH + 8 * g * VBL), tv1, x1);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          bool hi;
          const int j = pair_of_channel<VBL>(c, hi);
          fb[c][tp] = prmt(x0[j], x1[j], hi ? 0x7632u : 0x5410u);
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) mma16816(acc[mt], fa[mt][0], fb[mt][0], fa[mt][1], fb[mt][1], pb0, pb1);
    }
    __syncwarp();
    if (lane == 0 && !failed && i + kStages < my_pages) issue(i + kStages);
    __syncwarp();
  }

  // ---- combine the warps ----------------------------------------------------
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float l = l_run[c];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (g == 0) {
      red_m[warp][2 * t + c] = m_run[c];
      red_l[warp][2 * t + c] = l;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      red_acc[warp][2 * t + c][8 * g + mt] = acc[mt][c];
      red_acc[warp][2 * t + c][64 + 8 * g + mt] = acc[mt][c + 2];
    }
  }
  __syncthreads();
  const int j = threadIdx.x;
  for (int hh = 0; hh < a.G; ++hh) {
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][hh]);
    float lsum = 0.0f, A = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float sc = exp2f(red_m[w][hh] - M);
      lsum = fmaf(sc, red_l[w][hh], lsum);
      A = fmaf(sc, red_acc[w][hh][j], A);
    }
    float* dst = a.part + ((static_cast<long long>(b) * a.Hq + h * a.G + hh) * a.nchunks + chunk) * (kD + 2);
    if (j == 0) {
      dst[0] = M;
      dst[1] = lsum;
    }
    dst[2 + j] = A;
  }
}

template <int KBH, int KBL, int VBH, int VBL>
cudaError_t launch_combo(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.nchunks, a.H, a.B);
  if (a.kl.qjl)
    chunk_mma_kernel<KBH, KBL, VBH, VBL, true><<<grid, kThreads, 0, s>>>(a);
  else
    chunk_mma_kernel<KBH, KBL, VBH, VBL, false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

// Returns true (and the launch status in *err) when the configuration has a
// tensor-core kernel; false leaves the launch to the CUDA-core kernel.
bool launch_partials_mma(const DecodeArgs& a, cudaStream_t s, cudaError_t* err) {
  if (a.m != 128 || a.kl.split != 64 || a.vl.split != 64 || a.G > 8) return false;
  if ((reinterpret_cast<uintptr_t>(a.kc) | reinterpret_cast<uintptr_t>(a.vc)) & 15) return false;
  const int kh = a.kl.g[0].bits, kl = a.kl.g[1].bits, vh = a.vl.g[0].bits, vl = a.vl.g[1].bits;
  const int code = kh * 1000 + kl * 100 + vh * 10 + vl;
  switch (code) {
    case 3333: *err = launch_combo<3, 3, 3, 3>(a, s); return true;
    case 4343: *err = launch_combo<4, 3, 4, 3>(a, s); return true;
    case 3232: *err = launch_combo<3, 2, 3, 2>(a, s); return true;
    case 4444: *err = launch_combo<4, 4, 4, 4>(a, s); return true;
    case 2222: *err = launch_combo<2, 2, 2, 2>(a, s); return true;
    case 4422: *err = launch_combo<4, 4, 2, 2>(a, s); return true;
    default: return false;
  }
}

}  // namespace tq
