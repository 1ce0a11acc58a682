// Inner-product search on the tensor cores (tcgen05): the decode's two-stage
// score for 64 queries at a time against every database vector, and the k
// best per query kept on the way (no score array is written).
//
// [P2] "생각정리 209 (TurboQuant)": the vector-search use of the quantizer;
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §4.3: stage-1
// reconstruction plus the 1-bit QJL term estimates <q, x> without bias;
// §4.2: the codebook is only looked up.
//
// Per 128-vector tile (M = 128 database vectors, N = 64 queries, K = 128):
//   S1 = K^ Q~^T   K^ the stored codes' centroids as fp16 (a lookup table
//                  indexed by a byte of codes gives a centroid pair),
//   S2 = A  U^T    A = 1 + c b (fp16 1 or 1 + 255/1024 from sign bit b), so
//                  <u, 2b - 1> = (2/c) S2 - (2/c + 1) sum(u),
//   score = n16/sqrt(d) S1 + sqrt(pi/2)/m rho16 <u, 2b - 1>,
// the same fp16 operands the decode's partials kernel multiplies.
//
// One persistent CTA per SM, 14 warps (10 for 4-bit keys):
//   warp 0 (one lane): bulk copies of a tile's eight 16-vector key blocks into
//       a two-stage ring (page ids from the block table; an id out of range is
//       flagged and its vectors score -inf);
//   warp 1: tensor memory (256 columns: two slots of S1 | S2) and, one lane,
//       the MMAs of a tile once its operands are in shared memory;
//   warps 2-5: thread v builds row v of the two A tiles (fp16, 128-byte
//       swizzled K-major) from vector v's record, and its two score factors;
//   warps 6-13: two groups of four, group g taking the tiles of tensor-memory
//       slot g (every other tile), so one group's scan overlaps the other's
//       scores (4-bit keys: one group, warps 6-9; its lookup table leaves no
//       room for a second score tile); in a group, thread v reads row v (its vector) of S1 and S2,
//       writes the 64 scores to the group's shared tile; then thread 2q + h
//       scans query q's scores of vectors [64h, 64h + 64) and keeps its 16 best
//       (descending; a group sees its vectors in increasing index, so equal
//       scores keep the lower index).
// With two groups, group 0 merges the pair of lists of each (query, half) at
// the end.  search_merge_kernel then takes, per query, the k best of every
// CTA's lists
// (equal scores: lower index), and fills with -inf vectors in index order when
// fewer than k scores are finite.  With `scores` set the epilogue writes every
// score instead (the same arithmetic) and keeps no lists.
// Every wait is bounded; a wait that gives up sets the device error word and
// the CTA drains its copies and MMAs before it ends.

#include "tq_internal.h"
#include "tq_tc.cuh"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

using namespace tcx;

constexpr int kQB = 64;                 // queries per launch (MMA N)
constexpr int kTV = 128;                // database vectors per tile (MMA M)
constexpr int kTop = 16;                // list length per epilogue thread
constexpr int kWarpsFixed = 6;          // producer, MMA, four operand warps; then 4 or 8 epilogue warps
constexpr float kInvSqrtDS = 0.08838834764831845f;
constexpr float kSqrtHalfPiS = 1.2533141373155003f;
constexpr float kSignC = 255.0f / 1024.0f;
constexpr int kScoreRow = 136;          // floats per query row of the score tile (bank skew)
constexpr int kThrStride = 32;          // words between two queries' shared bars
constexpr int kThrBytes = kQB * kThrStride * 4;

// ---- codes ------------------------------------------------------------------
__host__ __device__ constexpr int lut_entries_s(int b) { return b == 4 ? 256 : b == 3 ? 120 : 16; }
__device__ __forceinline__ int stored_code_s(int b, int f) { return b == 4 ? (f < 8 ? f + 8 : 15 - f) : f; }
// 3-bit octet -> eight nibbles (channels 6 and 7 from the spare bit of each nibble).
__device__ __forceinline__ uint32_t octet_nibbles(uint32_t v) {
  return (v & 0x00777777u) | (((v & 0x00888888u) * 0x00204080u) & 0x77000000u);
}
// Bits [off, off + 32) of a little-endian word stream.
__device__ __forceinline__ uint32_t stream_bits(const uint32_t (&w)[17], int off) {
  return (off & 31) ? __funnelshift_r(w[off >> 5], w[(off >> 5) + 1], off & 31) : w[off >> 5];
}
// The four lookup indices of chunk cc (8 channels) of a group of B-bit codes
// starting at stream bit `base`: byte i = the index of channels (2i, 2i + 1).
template <int B>
__device__ __forceinline__ uint32_t chunk_index_bytes(const uint32_t (&w)[17], int base, int cc) {
  if (B == 4) return w[(base >> 5) + cc];
  if (B == 3) return octet_nibbles(stream_bits(w, base + 24 * cc));
  const uint32_t x = stream_bits(w, base + 16 * cc) & 0xFFFFu;   // 2-bit: nibble i -> byte i
  return (x & 0xFu) | ((x & 0xF0u) << 4) | ((x & 0xF00u) << 8) | ((x & 0xF000u) << 12);
}

struct TcSearchArgs {
  const float* qprep;        // [nq][d + m] fp32: q~ then u
  int nq, q0;                // this launch's queries: q0 .. q0 + min(64, nq - q0) - 1
  int n_db, num_pages, ntiles;
  const uint8_t* kc;
  const int32_t* bt;         // [ceil(n_db / 16)] page ids
  KindLayout kl;
  uint32_t* err;
  float2* cand;              // top-k lists of this launch: [gridDim.x][128][kTop] (score, index bits)
  float* scores;             // every score [nq][n_db] instead of lists (null: lists)
  unsigned* thr;             // [64][kThrStride] per query of this launch (one 128-byte line each, so the
                             // CTAs' atomics on different queries meet in different L2 slices): the
                             // largest k-th score any list has
                             // published, as an order-preserving key (0: none yet)
  int k;
};

// Order-preserving key of a float (larger float, larger key; -0 = +0); 0 is below every key.
__device__ __forceinline__ unsigned fkey(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? (f == 0.0f ? 0x80000000u : ~b) : (b | 0x80000000u);
}
__device__ __forceinline__ float funkey(unsigned u) {
  if (u == 0u) return -INFINITY;
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// c ? x : y, as a select instruction (opaque to the optimizer).
__device__ __forceinline__ float select_f(bool c, float x, float y) {
  float r;
  asm("{\n .reg .pred p;\n setp.ne.u32 p, %1, 0;\n selp.f32 %0, %2, %3, p;\n}" : "=f"(r)
      : "r"(static_cast<unsigned>(c)), "f"(x), "f"(y));
  return r;
}

// (score, index) ranks before (s2, i2): higher score, or equal score and lower
// index (an empty entry, index -1, last).
__device__ __forceinline__ bool better(float s, int i, float s2, int i2) {
  return s > s2 || (s == s2 && static_cast<unsigned>(i) < static_cast<unsigned>(i2));
}

// Shared memory (offsets from a 1024-aligned base); EG epilogue groups, a
// score tile each.
template <int EG>
struct SLayout {
  static constexpr int QH = 0;                       // q~ fp16 [64][128], swizzled
  static constexpr int UH = QH + kQB * 256;          // u fp16 [64][128]
  static constexpr int AK = UH + kQB * 256;          // K^ fp16 [128][128]
  static constexpr int AS = AK + kTV * 256;          // 1 + c b fp16 [128][128]
  static constexpr int SC = AS + kTV * 256;          // score tiles [2 groups][64][kScoreRow] fp32
  static constexpr int FAC = SC + EG * kQB * kScoreRow * 4;   // [4][256] fp32 score factors (ring)
  static constexpr int SU = FAC + 4 * 256 * 4;       // [64] -(2/c + 1) sum(u) per query
  static constexpr int PV = SU + kQB * 4;            // [4] page-valid masks
  static constexpr int BAR = PV + 16;                // mbarriers
  static constexpr int kRecFull = 0, kRecEmpty = 4, kAFull = 8, kAEmpty = 9, kTFull = 10, kTEmpty = 12,
                       kFacFull = 14, kNumBar = 18;
  static constexpr int TMEMA = BAR + 8 * kNumBar;
  static constexpr int REC = (TMEMA + 16 + 1023) & ~1023;   // ring of record stages (eight key blocks each)
};
constexpr int kSmemCapS = 232448;

template <int BH, int BL, bool QJL>
struct SGeo {
  static constexpr int CBK = 8 * (BH + BL);                           // code bytes per vector
  static constexpr int KBB = 16 * (CBK + (QJL ? 16 + 2 : 0) + 2);     // key block (16 vectors)
  static constexpr int K_SIGNS = 16 * CBK;
  static constexpr int K_NORM = K_SIGNS + (QJL ? 16 * 16 : 0);
  static constexpr int K_RNORM = K_NORM + 32;
  static constexpr int STAGE = 8 * KBB;
  static constexpr int E = lut_entries_s(BH) > lut_entries_s(BL) ? lut_entries_s(BH) : lut_entries_s(BL);
  // two epilogue groups when their second score tile fits next to a ring of at
  // least two record stages (the 4-bit lookup table is too large for it), then
  // the deepest ring (4, 3 or 2 stages) that fits; + 1024 alignment slack
  template <int eg>
  static constexpr int need(int st) { return ((SLayout<eg>::REC + st * STAGE + 1023) & ~1023) + 256 * E + 1024; }
  static constexpr int EG = need<2>(2) <= kSmemCapS ? 2 : 1;
  using L = SLayout<EG>;
  static constexpr int S = need<EG>(4) <= kSmemCapS ? 4 : need<EG>(3) <= kSmemCapS ? 3 : 2;
  static constexpr int NT = 32 * (kWarpsFixed + 4 * EG);   // threads per CTA
  static constexpr int LUT = (L::REC + S * STAGE + 1023) & ~1023;
  static constexpr int SMEM = LUT + 256 * E + 1024;
  static_assert(KBB % 16 == 0, "bulk copy unit");
  static_assert(SMEM <= kSmemCapS, "shared memory per block");
};

template <int BH, int BL, bool QJL>
__global__ void __launch_bounds__(SGeo<BH, BL, QJL>::NT, 1) search_tc_kernel(TcSearchArgs a) {
  using G = SGeo<BH, BL, QJL>;
  using L = typename G::L;
  constexpr int kThrS = G::NT;
  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char* sm = sm_raw + ((0u - su32(sm_raw)) & 1023u);
  const uint32_t sb = su32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto barx = [&](int i) { return sb + L::BAR + 8u * static_cast<uint32_t>(i); };
  const int nql = min(kQB, a.nq - a.q0);     // queries of this launch
  const int m = 128;

  // ---- setup: lookup tables, query operands, barriers, tensor memory --------
  {
    constexpr int E = G::E;
    for (int i = tid; i < E * 64; i += kThrS) {   // entry e, group g, lane l: the fp16 centroid pair
      const int l = i & 31, g = (i >> 5) & 1, e = i >> 6;
      const int b = g ? BL : BH;
      const GroupBook& gb = a.kl.g[g];
      uint32_t v = 0u;
      if (e < lut_entries_s(b)) {
        const int w = b == 2 ? 2 : 4, mask = b == 4 ? 15 : b == 3 ? 7 : 3;
        const __half lo = __float2half_rn(gb.c[stored_code_s(b, e & mask)]);
        const __half hi = __float2half_rn(gb.c[stored_code_s(b, (e >> w) & mask)]);
        v = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
      }
      *reinterpret_cast<uint32_t*>(sm + G::LUT + e * 256 + g * 128 + l * 4) = v;
    }
    // q~ and u rows of this launch as fp16 (zero rows past the last query); the
    // query prep (the kernel before this one) wrote them: wait for it here, after
    // the tables above were built
    pdl_wait();
    for (int i = tid; i < kQB * 32; i += kThrS) {        // (query, 8-channel chunk) of q~ and of u
      const int qr = i >> 5, c = i & 31, which = c >> 4, ch = c & 15;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if (qr < nql) {
        const float* src = a.qprep + static_cast<long long>(a.q0 + qr) * (kD + m) + (which ? kD : 0) + 8 * ch;
        const float4 f0 = *reinterpret_cast<const float4*>(src), f1 = *reinterpret_cast<const float4*>(src + 4);
        const __half2 h0 = __floats2half2_rn(f0.x, f0.y), h1 = __floats2half2_rn(f0.z, f0.w);
        const __half2 h2 = __floats2half2_rn(f1.x, f1.y), h3 = __floats2half2_rn(f1.z, f1.w);
        w[0] = *reinterpret_cast<const uint32_t*>(&h0), w[1] = *reinterpret_cast<const uint32_t*>(&h1);
        w[2] = *reinterpret_cast<const uint32_t*>(&h2), w[3] = *reinterpret_cast<const uint32_t*>(&h3);
      }
      sts128(sb + (which ? L::UH : L::QH) + chunk_off(qr, ch, kQB), w[0], w[1], w[2], w[3]);
    }
    if (tid < kQB) {   // -(2/c + 1) * sum of the fp16 u values the MMA multiplies
      float su = 0.0f;
      if (QJL && tid < nql) {
        const float* src = a.qprep + static_cast<long long>(a.q0 + tid) * (kD + m) + kD;
        for (int p = 0; p < m; ++p) su += __half2float(__float2half_rn(src[p]));
      }
      reinterpret_cast<float*>(sm + L::SU)[tid] = -(2.0f / kSignC + 1.0f) * su;
    }
    if (tid == 0) {
      for (int s = 0; s < 4; ++s) {
        bar_init(barx(L::kRecFull + s), 1);
        bar_init(barx(L::kRecEmpty + s), 4);
      }
      for (int s = 0; s < 2; ++s) {
        bar_init(barx(L::kTFull + s), 1);
        bar_init(barx(L::kTEmpty + s), 4);
      }
      bar_init(barx(L::kAFull), 4);
      bar_init(barx(L::kAEmpty), 1);
      for (int s = 0; s < 4; ++s) bar_init(barx(L::kFacFull + s), 4);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + L::TMEMA), "r"(256)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
  }
  const uint32_t tmem = *reinterpret_cast<const uint32_t*>(sm + L::TMEMA);
  int local = 0;
  if (static_cast<int>(blockIdx.x) < a.ntiles)
    local = (a.ntiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
  auto tile_of = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };
  bool failed = false;

  if (warp == 0) {
    // ---- producer (the whole warp): lane p < 8 holds the page id of page p of a
    // tile, loaded two tiles ahead; the lanes issue their pages' copies together
    constexpr int S = G::S;
    auto load_ids = [&](int i) {
      int pid = -1;
      if (i < local && lane < 8) {
        const int tp = tile_of(i) * kTV + 16 * lane;
        if (tp < a.n_db) pid = __ldg(a.bt + (tp >> 4));
      }
      return pid;
    };
    int id0 = load_ids(0), id1 = load_ids(1);
    int issued = 0;
    for (int i = 0; i < local; ++i) {
      const int s = i % S;
      const int pid = id0;
      id0 = id1;
      id1 = load_ids(i + 2);
      bool ok = true;
      if (lane == 0 && i >= S) ok = bar_wait(barx(L::kRecEmpty + s), ((i - S) / S) & 1, failed);
      if (!__shfl_sync(0xffffffffu, ok ? 1u : 0u, 0)) {
        failed = true;
        break;
      }
      const int t0 = tile_of(i) * kTV;
      const bool in_range = lane < 8 && t0 + 16 * lane < a.n_db;
      const bool valid = in_range && pid >= 0 && pid < a.num_pages;
      if (in_range && !valid) atomicOr(a.err, kErrPage);
      const uint32_t mask = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) {
        *reinterpret_cast<uint32_t*>(sm + L::PV + 4 * s) = mask;
        if (mask) bar_arrive_tx(barx(L::kRecFull + s), static_cast<uint32_t>(__popc(mask) * G::KBB));
        else bar_arrive(barx(L::kRecFull + s));
      }
      __syncwarp();
      if (valid) {
        fence_async_smem();
        g2s(sb + L::REC + s * G::STAGE + lane * G::KBB, a.kc + static_cast<long long>(pid) * G::KBB, G::KBB,
            barx(L::kRecFull + s));
      }
      issued = i + 1;
    }
    // copies still in flight land before the CTA ends
    if (lane == 0) {
      bool f2 = false;
      for (int j = issued >= S ? issued - S : 0; j < issued; ++j)
        (void)bar_wait(barx(L::kRecFull + j % S), (j / S) & 1, f2);
    }
  } else if (warp == 1) {
    // ---- MMA issue: the whole warp converged (conditions are warp votes), an elected lane
    // issuing each MMA and commit, so the operands stay in uniform registers ------------------
    {
      constexpr uint32_t id = idesc_f16(kQB);
      auto uni = [](bool x) { return __all_sync(0xffffffffu, x); };
      int done = 0;
      for (int i = 0; i < local; ++i) {
        const int slot = i & 1;
        if (!uni(bar_wait(barx(L::kAFull), i & 1, failed))) break;
        if (i >= 2 && !uni(bar_wait(barx(L::kTEmpty + slot), ((i - 2) >> 1) & 1, failed))) break;
        tc_after();
        const uint32_t d1 = tmem + 128u * slot, d2 = d1 + 64u;
#pragma unroll
        for (int k = 0; k < 8; ++k) mma_ss_warp(d1, kdesc(sb + L::AK, kTV, k), kdesc(sb + L::QH, kQB, k), id, k > 0);
        if (QJL) {
#pragma unroll
          for (int k = 0; k < 8; ++k) mma_ss_warp(d2, kdesc(sb + L::AS, kTV, k), kdesc(sb + L::UH, kQB, k), id, k > 0);
        }
        mma_commit_warp(barx(L::kAEmpty));
        mma_commit_warp(barx(L::kTFull + slot));
        done = i + 1;
      }
      bool f2 = false;
      if (done > 0) (void)bar_wait(barx(L::kTFull + ((done - 1) & 1)), ((done - 1) >> 1) & 1, f2);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---- operands: thread v builds row v of K^ and of the sign tile -------------
    const int v = tid - 64;
    const uint32_t lut = sb + G::LUT + static_cast<uint32_t>(lane) * 4u;
    for (int i = 0; i < local; ++i) {
      const int s = i % G::S;
      bool ok = bar_wait(barx(L::kRecFull + s), (i / G::S) & 1, failed);
      ok = ok && (i == 0 || bar_wait(barx(L::kAEmpty), (i - 1) & 1, failed));
      if (!__all_sync(0xffffffffu, ok)) {                // the warp gives up together
        failed = true;
        break;
      }
      const uint32_t mask = *reinterpret_cast<const uint32_t*>(sm + L::PV + 4 * s);
      const int t = tile_of(i) * kTV + v;
      const bool valid = (mask >> (v >> 4) & 1u) && t < a.n_db;
      float fa = __int_as_float(0x7FC00000), fb = 0.0f;   // NaN factor: no score for this row
      if (valid) {
        const uint32_t blk = sb + L::REC + s * G::STAGE + (v >> 4) * G::KBB;   // stage s = i % S
        const int slot = v & 15;
        uint32_t w[17];
#pragma unroll
        for (int k = 0; k < G::CBK / 8; ++k) {
          const uint2 x = lds64(blk + slot * G::CBK + 8 * k);
          w[2 * k] = x.x;
          w[2 * k + 1] = x.y;
        }
#pragma unroll
        for (int k = G::CBK / 4; k < 17; ++k) w[k] = 0u;
        // K^ row: chunk c = channels 8c .. 8c + 7
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int g = c >> 3, cc = c & 7;
          const uint32_t x = g ? chunk_index_bytes<BL>(w, 64 * BH, cc) : chunk_index_bytes<BH>(w, 0, cc);
          const uint32_t lb = lut + (g ? 128u : 0u);
          const uint32_t p0 = lds32(prmt(x, 0, 0x4404u) + lb);
          const uint32_t p1 = lds32(prmt(x, 0, 0x4414u) + lb);
          const uint32_t p2 = lds32(prmt(x, 0, 0x4424u) + lb);
          const uint32_t p3 = lds32(prmt(x, 0, 0x4434u) + lb);
          sts128(sb + L::AK + chunk_off(v, c, kTV), p0, p1, p2, p3);
        }
        if (QJL) {
          // sign tile row: byte c of the sign bits -> projections 8c .. 8c + 7 as (1 + c b) pairs
          const uint4 sw = lds128(blk + G::K_SIGNS + slot * 16);
          const uint32_t sws[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint32_t byte = (sws[c >> 2] >> (8 * (c & 3))) & 0xFFu;
            // bits 0-3 (then 4-7) to the top bit of bytes 0-3: prmt's sign replication
            // turns each into 0xFF or 0 under a 0x3C high byte (fp16 1 or 1 + c)
            const uint32_t zl = ((byte & 0xFu) * 0x10204080u) & 0x80808080u;
            const uint32_t zh = ((byte >> 4) * 0x10204080u) & 0x80808080u;
            sts128(sb + L::AS + chunk_off(v, c, kTV), prmt(zl, 0x3C3C3C3Cu, 0x4948u), prmt(zl, 0x3C3C3C3Cu, 0x4B4Au),
                   prmt(zh, 0x3C3C3C3Cu, 0x4948u), prmt(zh, 0x3C3C3C3Cu, 0x4B4Au));
          }
          fb = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(blk + G::K_RNORM + 2 * slot)))) *
               (kSqrtHalfPiS / m);
        }
        fa = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(blk + G::K_NORM + 2 * slot)))) * kInvSqrtDS;
      }
      const uint32_t fac = sb + L::FAC + (i & 3) * 1024;
      stsf(fac + 4 * v, fa);
      stsf(fac + 512 + 4 * v, fb);
      fence_async_smem();                      // the operand rows, for the tensor cores
      __syncwarp();
      if (lane == 0) {
        bar_arrive(barx(L::kAFull));
        bar_arrive(barx(L::kRecEmpty + s));
        bar_arrive(barx(L::kFacFull + (i & 3)));
      }
    }
  } else {
    // ---- epilogue ---------------------------------------------------------------
    // G::EG groups of four warps, group eg taking the tiles i = eg, eg + EG, ...
    // (with two groups, group eg has tensor-memory slot eg)
    const int eg = (warp - 6) >> 2;
    const int wq = warp & 3, v = 32 * wq + lane;       // tensor-memory lanes 32 wq .. : vector v
    const int tl = (tid - 192) & 127;                    // 0 .. 127 within the group
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * wq) << 16);
    const uint32_t sc = sb + L::SC + eg * (kQB * kScoreRow * 4);
    const uint32_t su = sb + L::SU;
    float best[kTop];
    int bidx[kTop];
#pragma unroll
    for (int j = 0; j < kTop; ++j) best[j] = -INFINITY, bidx[j] = -1;
    const int sq = tl >> 1, sh = tl & 1;                 // scan: query sq, vectors [64 sh, 64 sh + 64)
    float kth = -INFINITY;                               // this list's k-th best (its insertion bar)
    unsigned published = 0u;
    for (int i = eg; i < local; i += G::EG) {
      const int slot = i & 1;
      // a wait that gives up leaves this tile's results undefined (the error word
      // says so) but the loop goes on, so the named barriers below are still met
      // the shared bar of this thread's scan query, read early (an L2 round trip)
      unsigned gkey = 0u;
      if (!a.scores)   // volatile: issued here, not sunk to its first use
        asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(gkey) : "l"(a.thr + kThrStride * sq) : "memory");
      bool ok = bar_wait(barx(L::kFacFull + (i & 3)), (i >> 2) & 1, failed);
      const uint32_t fac = sb + L::FAC + (i & 3) * 1024;
      const float fa = ldsf(fac + 4 * v), fb = ldsf(fac + 512 + 4 * v);
      ok = bar_wait(barx(L::kTFull + slot), (i >> 1) & 1, failed) && ok;
      if (!__all_sync(0xffffffffu, ok)) failed = true;
      tc_after();
      const int t0 = tile_of(i) * kTV;
      const bool has = !isnan(fa);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {                      // queries 32h .. 32h + 31 (rolled, as below: smaller
                                                         // epilogue code for the instruction cache)
        float s1[32], s2[32];
        tld32(trow + 128u * slot + 32u * h, s1);
        if (QJL) tld32(trow + 128u * slot + 64u + 32u * h, s2);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int qq = 32 * h + k;
          const float q2 = QJL ? fmaf(2.0f / kSignC, s2[k], ldsf(su + 4 * qq)) : 0.0f;
          s1[k] = has ? fmaf(fa, s1[k], fb * q2) : -INFINITY;
        }
        if (a.scores) {
          const int t = t0 + v;
          if (t < a.n_db) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (32 * h + k < nql) a.scores[static_cast<long long>(a.q0 + 32 * h + k) * a.n_db + t] = s1[k];
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) stsf(sc + 4 * ((32 * h + k) * kScoreRow + v + (v >= 64 ? 4 : 0)), s1[k]);
        }
      }
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(barx(L::kTEmpty + slot));
      if (!a.scores) {
        nsync(1 + eg, 128);                              // the tile's scores are in
        const uint32_t row = sc + 4 * (sq * kScoreRow + 68 * sh);
        const int tb = t0 + 64 * sh;
        // a score below the largest published k-th score of this query cannot be in
        // the answer (that list's k best are candidates); equal ones still can
        const float gt = funkey(gkey);
        // while the list is short of k entries: the k-th largest of the 16 group
        // maxima is at most this tile's k-th best (k distinct elements reach it),
        // so an element below it cannot be among the list's final k (taken first,
        // so that pass 1 marks only the elements over it)
        float bar0 = -INFINITY;
        if (kth == -INFINITY) {                          // (rare: the first tiles) the tile twice
          float gmax[16];
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const uint4 xu = lds128(row + 4 * j);
            gmax[j >> 2] = fmaxf(fmaxf(__uint_as_float(xu.x), __uint_as_float(xu.y)),
                                 fmaxf(__uint_as_float(xu.z), __uint_as_float(xu.w)));
          }
#pragma unroll 1
          for (int g = 0; g < 16; ++g) {
            int ge = 0;
#pragma unroll
            for (int h = 0; h < 16; ++h) ge += gmax[h] >= gmax[g] ? 1 : 0;
            if (ge >= a.k) bar0 = fmaxf(bar0, gmax[g]);
          }
        }
        // pass 1 (every lane, no branches): the elements over the bar, as a bit mask;
        // while the list is short, the bar is bar0 (the list's own is -inf then)
        const bool use_gt = gt > kth;
        const float bar = use_gt ? gt : kth;
        uint32_t mlo = 0u, mhi = 0u;
        if (bar0 > -INFINITY) {
          const float b0 = fmaxf(bar0, gt);
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const uint4 xu = lds128(row + 4 * j);
            const float xv[4] = {__uint_as_float(xu.x), __uint_as_float(xu.y), __uint_as_float(xu.z),
                                 __uint_as_float(xu.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t bit = xv[e] >= b0 ? 1u : 0u;
              if (j + e < 32) mlo |= bit << (j + e);
              else mhi |= bit << (j + e - 32);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const uint4 xu = lds128(row + 4 * j);
            const float xv[4] = {__uint_as_float(xu.x), __uint_as_float(xu.y), __uint_as_float(xu.z),
                                 __uint_as_float(xu.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t bit = (use_gt ? xv[e] >= bar : xv[e] > bar) ? 1u : 0u;
              if (j + e < 32) mlo |= bit << (j + e);
              else mhi |= bit << (j + e - 32);
            }
          }
        }
        // pass 2: the (few) marked elements in index order; the warp loops only as
        // often as its busiest lane
        while (mlo | mhi) {
          const int e = mlo ? __ffs(mlo) - 1 : 31 + __ffs(mhi);
          if (mlo) mlo &= mlo - 1u;
          else mhi &= mhi - 1u;
          const float cs = ldsf(row + 4 * e);
          if (!(cs > kth && cs >= gt && cs >= bar0)) continue;   // the bar rose since pass 1
          const int ci = tb + e;
          // insert at position p = #entries >= cs (equal scores keep the earlier, lower
          // index ahead); cs > kth puts p below k; the shift is one parallel step
          int p = 0;
#pragma unroll
          for (int r = 0; r < kTop; ++r) p += best[r] >= cs ? 1 : 0;
#pragma unroll
          for (int r = kTop - 1; r > 0; --r) {
            best[r] = r > p ? best[r - 1] : (r == p ? cs : best[r]);
            bidx[r] = r > p ? bidx[r - 1] : (r == p ? ci : bidx[r]);
          }
          if (p == 0) best[0] = cs, bidx[0] = ci;
          // the k-th entry by selects the compiler cannot fold into an indexed load
          // (an index would move the list to local memory)
#pragma unroll
          for (int r = 0; r < kTop; ++r) kth = select_f(r == a.k - 1, best[r], kth);
        }
        if (kth > -INFINITY && fkey(kth) > published) {  // share this list's k-th best
          published = fkey(kth);
          atomicMax(a.thr + kThrStride * sq, published);
        }
        nsync(1 + eg, 128);                              // before the next tile's scores
      }
    }
    if (!a.scores) {
      float2* out = a.cand + (static_cast<long long>(blockIdx.x) * kTV + tl) * kTop;
      if (G::EG == 1) {
#pragma unroll
        for (int j = 0; j < kTop; ++j) out[j] = make_float2(best[j], __int_as_float(bidx[j]));
      } else {
        // the two groups' lists of this (query, half) merged into one (the merge
        // kernel then reads one list per (query, half) and CTA): each group puts
        // its list in its own score tile, group 0 merges the pair
        float2* mine = reinterpret_cast<float2*>(sm + L::SC + eg * (kQB * kScoreRow * 4)) + tl * kTop;
#pragma unroll
        for (int j = 0; j < kTop; ++j) mine[j] = make_float2(best[j], __int_as_float(bidx[j]));
        nsync(3, 256);
        if (eg == 0) {
          const float2* other = reinterpret_cast<const float2*>(sm + L::SC + kQB * kScoreRow * 4) + tl * kTop;
          int ia = 0, ib = 0;
          for (int j = 0; j < kTop; ++j) {
            const float2 x = mine[ia], y = other[ib];
            const bool take_a = ib >= kTop ||
                                (ia < kTop && !better(y.x, __float_as_int(y.y), x.x, __float_as_int(x.y)));
            out[j] = take_a ? x : y;
            ia += take_a ? 1 : 0;
            ib += take_a ? 0 : 1;
          }
        }
      }
    }
  }
  if (failed) atomicOr(a.err, kErrTimeout);
  pdl_trigger();                                         // the merge may be launched (it waits for this grid)
  tc_before();
  __syncthreads();
  tc_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256) : "memory");
}

// ---- merge: the k best of every CTA's lists, one warp per query ----------------

// The merge's buffer holds every entry of every list (when all tie): 2 lists of
// 16 per query in each of the grid CTAs (a CTA's two epilogue groups merged).
size_t merge_smem_bytes(int groups) { return sizeof(float2) * 2 * static_cast<size_t>(groups) * kTop; }

// Launched after the scoring kernel of queries q0 .. q0 + gridDim.x - 1, one
// block of sixteen warps per query (a thread loads one whole list at once).  tau, the largest k-th score over the lists,
// is at most the answer's k-th score (that list's k best are candidates), so
// only entries >= tau can be in the answer; they are gathered (usually a little
// over k), then sorted by (score descending, index ascending) -- by warp 0 in
// registers when 32 or fewer, else by k rounds of selection.
constexpr int kMergeThreads = 512;   // 16 warps: one or two lists per thread, loads in one round
__global__ void __launch_bounds__(kMergeThreads) search_merge_kernel(const float2* cand, int grid, int q0, int n_db,
                                                                    int k, float* top_s, int32_t* top_i) {
  extern __shared__ float2 buf[];                        // 2 grid kTop entries
  const int kMergeBuf = 2 * grid * kTop;
  __shared__ float wmax[kMergeThreads / 32];
  __shared__ int nbuf;
  const int ql = blockIdx.x, q = q0 + ql, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nl = 2 * grid;                               // list l: thread 2 ql + (l & 1) of CTA l / 2
  auto list = [&](int l) {
    return cand + (static_cast<long long>(l >> 1) * kTV + 2 * ql + (l & 1)) * kTop;
  };
  if (tid == 0) nbuf = 0;
  pdl_wait();                                            // the scoring kernel's lists
  auto gather = [&](const float4 (&x)[kTop / 2], float tau) {
#pragma unroll
    for (int j = 0; j < kTop / 2; ++j) {
      if (__float_as_int(x[j].y) >= 0 && x[j].x >= tau) {
        const int at = atomicAdd(&nbuf, 1);
        if (at < kMergeBuf) buf[at] = make_float2(x[j].x, x[j].y);
      }
      if (__float_as_int(x[j].w) >= 0 && x[j].z >= tau) {
        const int at = atomicAdd(&nbuf, 1);
        if (at < kMergeBuf) buf[at] = make_float2(x[j].z, x[j].w);
      }
    }
  };
  auto block_max = [&](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) wmax[warp] = v;
    __syncthreads();
    v = wmax[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) v = fmaxf(v, wmax[w]);
    return v;
  };
  if (nl <= kMergeThreads) {
    // one list per thread at most: the whole list in one batch of loads, tau from
    // the registers, then the entries >= tau
    float4 x[kTop / 2];
    float t = -INFINITY;
    if (tid < nl) {
      const float4* src = reinterpret_cast<const float4*>(list(tid));
#pragma unroll
      for (int j = 0; j < kTop / 2; ++j) x[j] = src[j];
#pragma unroll
      for (int j = 0; j < kTop / 2; ++j) {               // entry k - 1: x[(k-1)/2], half (k-1)&1
        if (2 * j == k - 1 && __float_as_int(x[j].y) >= 0) t = x[j].x;
        if (2 * j + 1 == k - 1 && __float_as_int(x[j].w) >= 0) t = x[j].z;
      }
    }
    const float tau = block_max(t);
    if (tid < nl) gather(x, tau);
  } else {
    float t = -INFINITY;
#pragma unroll 4
    for (int l = tid; l < nl; l += kMergeThreads) {
      const float2 e = list(l)[k - 1];
      if (__float_as_int(e.y) >= 0) t = fmaxf(t, e.x);
    }
    const float tau = block_max(t);
#pragma unroll 2
    for (int l = tid; l < nl; l += kMergeThreads) {
      const float4* src = reinterpret_cast<const float4*>(list(l));
      float4 x[kTop / 2];
#pragma unroll
      for (int j = 0; j < kTop / 2; ++j) x[j] = src[j];   // the whole list in one batch of loads
      gather(x, tau);
    }
  }
  __syncthreads();
  if (warp != 0) return;
  const int count = nbuf < kMergeBuf ? nbuf : kMergeBuf;
  int chosen[kTop];
  int found = 0;
  if (count <= 32) {
    float sv = -INFINITY;
    int iv = 0x7FFFFFFF;
    if (lane < count) sv = buf[lane].x, iv = __float_as_int(buf[lane].y);
    // bitonic sort across the warp, best first
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, sv, stride);
        const int io = __shfl_xor_sync(0xffffffffu, iv, stride);
        const bool lower = (lane & stride) == 0;
        const bool desc = (lane & size) == 0;            // this block sorts best first
        const bool other_better = better(so, io, sv, iv);
        if (lower == desc ? other_better : !other_better && !(so == sv && io == iv)) sv = so, iv = io;
      }
    }
    found = count < k ? count : k;
    if (lane < found) {
      top_s[static_cast<long long>(q) * k + lane] = sv;
      top_i[static_cast<long long>(q) * k + lane] = iv;
    }
#pragma unroll
    for (int r = 0; r < kTop; ++r) chosen[r] = __shfl_sync(0xffffffffu, iv, r);
  } else {
    for (int r = 0; r < k; ++r) {
      float sv = -INFINITY;
      int iv = 0x7FFFFFFF, at = -1;
      for (int j = lane; j < count; j += 32) {
        const float2 e = buf[j];
        const int ie = __float_as_int(e.y);
        if (ie >= 0 && better(e.x, ie, sv, iv)) sv = e.x, iv = ie, at = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, sv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, iv, o);
        const int a2 = __shfl_xor_sync(0xffffffffu, at, o);
        if (better(s2, i2, sv, iv)) sv = s2, iv = i2, at = a2;
      }
      if (at < 0) break;
      if (lane == 0) {
        top_s[static_cast<long long>(q) * k + r] = sv;
        top_i[static_cast<long long>(q) * k + r] = iv;
        buf[at].y = __int_as_float(-1);                  // taken
      }
      __syncwarp();
      chosen[r] = iv;
      found = r + 1;
    }
  }
  // fewer than k finite scores: every other vector scores -inf; the lowest indices follow
  if (lane == 0 && found < k) {
    int r = found;
    for (int t = 0; t < n_db && r < k; ++t) {
      bool used = false;
      for (int j = 0; j < found; ++j) used = used || chosen[j] == t;
      if (used) continue;
      top_s[static_cast<long long>(q) * k + r] = -INFINITY;
      top_i[static_cast<long long>(q) * k + r] = t;
      ++r;
    }
  }
}

// The merge kernel's shared memory, set once per device for the largest grid
// (one CTA per SM).
cudaError_t merge_attr(int grid) {
  static std::atomic<unsigned long long> configured{0};
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (grid > sms) return cudaErrorInvalidValue;
  return smem_attr_once(search_merge_kernel, static_cast<int>(merge_smem_bytes(sms)), configured);
}

// Per 64 queries: the scoring kernel, then (lists) the merge of its lists.
template <int BH, int BL, bool QJL>
cudaError_t launch_tc(const TcSearchArgs& base, int grid, int k, float* top_s, int32_t* top_i, cudaStream_t st) {
  using G = SGeo<BH, BL, QJL>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = smem_attr_once(search_tc_kernel<BH, BL, QJL>, G::SMEM, configured);
  if (e != cudaSuccess) return e;
  if ((e = merge_attr(grid)) != cudaSuccess) return e;
  for (int q0 = 0; q0 < base.nq; q0 += kQB) {
    TcSearchArgs a = base;
    a.q0 = q0;
    a.k = k;
    if (q0 > 0 && !a.scores && (e = cudaMemsetAsync(a.thr, 0, kThrBytes, st)) != cudaSuccess)
      return e;   // (the first block's bars are cleared before the query prep)
    if ((e = launch_pdl(search_tc_kernel<BH, BL, QJL>, dim3(grid), dim3(G::NT), static_cast<size_t>(G::SMEM), st, a)) !=
        cudaSuccess)
      return e;
    if (!a.scores) {
      const int nql = base.nq - q0 < kQB ? base.nq - q0 : kQB;
      if ((e = launch_pdl(search_merge_kernel, dim3(nql), dim3(kMergeThreads), merge_smem_bytes(grid), st,
                          static_cast<const float2*>(a.cand), grid, q0, a.n_db, k, top_s, top_i)) != cudaSuccess)
        return e;
    }
  }
  return cudaSuccess;
}

template <int BH, int BL>
cudaError_t launch_tc_q(const TcSearchArgs& a, int grid, int k, float* top_s, int32_t* top_i, cudaStream_t st) {
  return a.kl.qjl ? launch_tc<BH, BL, true>(a, grid, k, top_s, top_i, st)
                  : launch_tc<BH, BL, false>(a, grid, k, top_s, top_i, st);
}

int tc_grid(int ntiles) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return ntiles < sms ? ntiles : sms;
}

}  // namespace

bool search_tc_supported(const KindLayout& kl, int m, int k_top) {
  if (m != 128 || kl.split != 64 || k_top > kTop) return false;
  for (int g = 0; g < 2; ++g)
    if (kl.g[g].bits < 2 || kl.g[g].bits > 4) return false;
  return true;
}

size_t search_tc_cand_bytes() {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sizeof(float2) * static_cast<size_t>(sms) * kTV * kTop + kThrBytes;   // the CTAs' lists, the bars
}

cudaError_t launch_search_tc(const DecodeArgs& qa, const uint8_t* kc, const int32_t* bt, int num_pages, int n_db,
                             int k, float* top_s, int32_t* top_i, float* scores, void* cand, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (!scores) {   // the shared per-query bars of the first 64 queries start at "none"
    e = cudaMemsetAsync(static_cast<char*>(cand) + search_tc_cand_bytes() - kThrBytes, 0, kThrBytes, st);
    if (e != cudaSuccess) return e;
  }
  e = launch_decode(qa, TQ_STAGE_QPREP, st);
  if (e != cudaSuccess) return e;
  TcSearchArgs a{};
  a.qprep = qa.qprep;
  a.nq = qa.B * qa.Hq;
  a.q0 = 0;
  a.n_db = n_db;
  a.num_pages = num_pages;
  a.ntiles = (n_db + kTV - 1) / kTV;
  a.kc = kc;
  a.bt = bt;
  a.kl = qa.kl;
  a.err = qa.tab.err;
  a.cand = scores ? nullptr : static_cast<float2*>(cand);
  a.thr = scores ? nullptr
                 : reinterpret_cast<unsigned*>(static_cast<char*>(cand) + search_tc_cand_bytes() - kThrBytes);
  a.scores = scores;
  const int grid = tc_grid(a.ntiles);
  switch (qa.kl.g[0].bits * 10 + qa.kl.g[1].bits) {
    case 22: return launch_tc_q<2, 2>(a, grid, k, top_s, top_i, st);
    case 23: return launch_tc_q<2, 3>(a, grid, k, top_s, top_i, st);
    case 24: return launch_tc_q<2, 4>(a, grid, k, top_s, top_i, st);
    case 32: return launch_tc_q<3, 2>(a, grid, k, top_s, top_i, st);
    case 33: return launch_tc_q<3, 3>(a, grid, k, top_s, top_i, st);
    case 34: return launch_tc_q<3, 4>(a, grid, k, top_s, top_i, st);
    case 42: return launch_tc_q<4, 2>(a, grid, k, top_s, top_i, st);
    case 43: return launch_tc_q<4, 3>(a, grid, k, top_s, top_i, st);
    default: return launch_tc_q<4, 4>(a, grid, k, top_s, top_i, st);
  }
}

}  // namespace tq
