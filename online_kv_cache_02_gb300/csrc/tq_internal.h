// Internal declarations shared by the library's translation units.
#ifndef TQ_INTERNAL_H_
#define TQ_INTERNAL_H_

#include "../../include/tq.h"

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace tq {

constexpr int kD = 128;          // supported head dimension
constexpr int kPage = 16;        // tokens per cache page
constexpr int kMaxM = 128;       // QJL projections, multiple of 32
constexpr int kMaxGroup = 8;     // query heads per KV head handled by the decode kernels
constexpr float kPiScale = 16.0f;  // Pi is split into fp16 hi + lo after scaling by this power of two
constexpr int kQFragWords = 192;   // query fragment words per query row (see DecodeArgs::qfrag)

// Device error word bits.
constexpr uint32_t kErrPage = 1u;      // page id outside [0, num_pages)
constexpr uint32_t kErrBlock = 2u;     // position beyond the block table
constexpr uint32_t kErrSeqLen = 4u;    // sequence length beyond max_seq_len / block table
constexpr uint32_t kErrTimeout = 8u;   // a bounded wait gave up
constexpr uint32_t kErrLayout = 16u;   // shared-memory layout did not fit

// One channel group's Lloyd-Max codebook in unit-variance units.
struct GroupBook {
  int bits;
  int nb;                // 2^bits - 1 boundaries
  float c[16];           // centroids, fp32
  float c_lo[16];        // c64 - c (double-float low parts)
  float t[16];           // boundaries, fp32 (entries >= nb are +inf)
  double c64[16];
  double t64[16];
};

// Codebooks and bit layout for one kind (K or V).
struct KindLayout {
  GroupBook g[2];        // g[0]: channels [0, split), g[1]: [split, d)
  int split;
  int code_bytes;        // per vector
  int block_bytes;       // per (page, head) block
  int off_signs;         // byte offsets inside a block
  int off_norm;
  int off_rnorm;
  int qjl;               // keys with QJL signs + residual norm
};

// Key channel pairing of the persistent decode kernel: thread slice t covers
// channels 16t..16t+15 of a channel group; pair j (0..7) holds the channel
// below plus the next one (see tq_decode_lut.cu).  Shared with qprep, which
// writes the query fragments in this order.
__host__ __device__ constexpr int k_pair_channel(int b, int j) {
  return b == 2 ? (j < 4 ? 4 * j : 4 * (j - 4) + 2) : 2 * j;
}

// Host functions (tq_host.cpp).
void gaussian_fill(uint64_t seed, uint64_t stream, size_t n, double* out);
void rotation_fill(int d, uint64_t seed, double* pi);
void qjl_fill(int m, int d, uint64_t seed, double* s);
void codebook_fill(int bits, double* centroids, double* boundaries);
void codebook_fill_sphere(int bits, int d, double* centroids, double* boundaries);

// Device tables owned by a context.
struct DeviceTables {
  float* pit;            // Pi^T, fp32 [d][d]: pit[k*d + i] = Pi[i][k]
  float* pi;             // Pi, fp32 [d][d] row-major
  double* pi64;          // Pi, fp64 row-major
  float* st;             // S^T, fp32 [d][m]: st[j*m + i] = S[i][j]
  double* s64;           // S, fp64 row-major [m][d]
  uint32_t* err;         // device error word
  unsigned long long* counters;  // [0] codes re-taken in fp64, [1] sign bits re-taken
  // tensor-core quantize operands: fp16 bit patterns in the 128-byte-swizzled
  // K-major layout (rows of 64 channels per 128 B, chunk index XOR row % 8,
  // two 64-channel halves one after the other)
  unsigned short* pih_sw;   // Pi rounded to fp16, [128 rows][128]
  unsigned short* pil_sw;   // fp16(Pi - pih)
  unsigned short* sh_sw;    // S rounded to fp16, [m rows][128]
  unsigned short* sl_sw;    // fp16(S - sh)
  float* a_df;              // (S Pi) as double-float pairs [m][128][2]
  float* s_df;              // S as double-float pairs [m][128][2]
  float* pi_df;             // Pi as double-float pairs [128][128][2]
  float* wt;                // W^T, fp32 [d][d + m]: W = [Pi; S Pi], wt[k*(d+m) + r] = W[r][k]
};

struct QuantizeArgs {
  const void* x;         // [batch][n_new][H][d]
  int f32;               // 1: fp32 input, 0: bf16
  int batch, n_new, H;
  const int32_t* start_pos;
  const int32_t* block_table;
  int maxp, num_pages;
  uint8_t* cache;
  long long page_bytes;
  int m;
  KindLayout lay;
  DeviceTables tab;
  int max_ctas;          // 0: up to one CTA per SM; else at most this many
};

struct DecodeArgs {
  const void* q;
  int f32;
  int B, Hq, H, G;
  const int32_t* seq_lens;
  int len_add;           // tokens appended in the same call (added to seq_lens[b])
  int max_seq_len;
  const int32_t* block_table;
  int maxp, num_pages;
  const uint8_t* kc;
  const uint8_t* vc;
  long long k_page_bytes, v_page_bytes;
  int chunk, nchunks;
  float scale_log2;      // softmax_scale * log2(e)
  int m;
  KindLayout kl, vl;
  DeviceTables tab;
  float* qprep;          // [B][Hq][d + m]
  float* part;           // [B][Hq][nchunks][d + 2]
  float* out;            // [B][Hq][d]
  int* sched;            // [2] work counter and finished-warp count of the persistent kernel (zeroed by qprep)
  int chained;           // 1: qprep follows the fused step's append kernel (a dependent launch that
                         // overlaps it and waits for it before finishing, so the partials kernel sees
                         // the new token in the cache)
  int max_ctas;          // partials kernel: 0 = one CTA per SM, else at most this many
  uint32_t* qfrag;       // [B][Hq][kQFragWords] fp16 pairs in the persistent kernel's fragment order (m = 128
                         // only): words 32 t .. 32 t + 31 for lane t%4 of a KV-head warp (16 of q~ key pairs, 16
                         // of u), then 128 + 16 t .. : the fp16 low parts of lane t's q~ pairs
  // causal attention of T > 0 new tokens per sequence (0: decode): the query
  // rows are [B][T][Hq] (qprep, partials and out use B * T rows), seq_lens
  // holds each sequence's first new position, len_add = T, and the partials
  // kernel takes query rows eight at a time (nqb blocks per sequence and KV head)
  int T;
  int nqb;
  // 1: qprep writes each row as fp16 words in tensor-memory column order
  // (64 of q~ hi pairs, 64 of q~ lo pairs, 64 of u pairs) for the tensor-core
  // causal kernel, instead of the fp32 [q~; u]
  int qhalf;
};

// Opt kernel `fn` into `bytes` of dynamic shared memory on the current device,
// once per device: `done` (one static per launch site) keeps a bit per device
// ordinal below 64 (higher ordinals set the attribute on every call).  Safe to
// call from several host threads: setting the attribute twice is harmless.
template <typename Kernel>
cudaError_t smem_attr_once(Kernel* fn, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Programmatic dependent launch: a kernel launched this way may start while the
// previous kernel of the stream still runs; it calls pdl_wait() before it reads
// anything that kernel writes (griddepcontrol.wait returns once the previous
// grid has completed and its memory is visible).  pdl_trigger() lets the next
// such kernel launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s);
// One warp per vector (a decode step's new tokens): false if the shapes are not taken.
bool launch_append(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err);
// Tensor-core quantize of K and V in one launch (bf16 inputs, supported
// bit-width combinations); returns false when the configuration is not covered.
bool launch_quantize_tc(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err);
// Pipelined tensor-core quantize of bf16 K and V (tq_quantize_pipe.cu): TMA
// x tiles, bf16 MMAs, warp-specialized epilogue; any bit widths 1-4 and
// splits that are multiples of 32.  Returns false when the inputs are not
// covered (fp32 inputs, a codebook too fine for its cell tables).
bool launch_quantize_pipe(const QuantizeArgs& k, const QuantizeArgs& v, cudaStream_t s, cudaError_t* err);
cudaError_t launch_decode(const DecodeArgs& a, int stages, cudaStream_t s);
// Head dimensions other than 128 (tq_generic.cu): CUDA-core quantize and
// decode for d a multiple of 32 up to 256.
constexpr int kDMax = 256;
cudaError_t launch_quantize_generic(const QuantizeArgs& a, int d, cudaStream_t s);
cudaError_t launch_decode_generic(const DecodeArgs& a, int d, int stages, cudaStream_t s);
// Persistent lookup-table kernel (tq_decode_lut.cu): CTAs it runs with at
// most, one per SM (0: configuration not supported), and its launch (false:
// not supported).  A launch runs 12 or 16 warps per CTA: every warp takes
// whole split-K items (chunks of one KV head) from a shared counter, a warp's
// speed scales as 1/warps per CTA, so lut_cost (waves of items over the warp
// slots x per-item cost x warps) estimates the time and lut_warps_for picks
// the cheaper count.
int lut_decode_ctas(const KindLayout& kl, const KindLayout& vl, int m, int G);
long long lut_cost(long long items, int ctas, int warps, long long chunk_cost);
int lut_warps_for(long long items, int ctas);
// Inner-product search on CUDA cores (tq_search.cu): bytes of the q~/u rows;
// the launches (qprep of qa, scores into `scores`, then the top k unless
// top_s is null) and the largest k supported.
size_t search_qrows_bytes(int nq, int m);
cudaError_t launch_search(const DecodeArgs& qa, const uint8_t* kc, const int32_t* bt, int num_pages, int n_db,
                          int k, float* top_s, int32_t* top_i, float* scores, cudaStream_t st);
int search_max_k();
int search_max_queries();
// Inner-product search on the tensor cores (tq_search_tc.cu): whether the
// configuration and k take that path, the bytes of its per-CTA candidate
// lists, and the launches (qprep of qa, the scoring kernel per 64 queries,
// then the merge into the top k; with `scores` set, every score instead).
bool search_tc_supported(const KindLayout& kl, int m, int k_top);
size_t search_tc_cand_bytes();
cudaError_t launch_search_tc(const DecodeArgs& qa, const uint8_t* kc, const int32_t* bt, int num_pages, int n_db,
                             int k, float* top_s, int32_t* top_i, float* scores, void* cand, cudaStream_t st);
bool launch_partials_lut(const DecodeArgs& a, cudaStream_t s, cudaError_t* err);
// Causal attention on the tensor cores (tq_causal_tc.cu): query rows per
// block (the MMA's M), the largest chunk, whether the configuration takes
// that path, and the partials launch over B x H x query blocks x chunks items
// (qprep before it, the merge after it, as for the decode).
int causal_tc_block_rows();
int causal_tc_max_chunk();
bool causal_tc_supported(const KindLayout& kl, const KindLayout& vl, int m);
cudaError_t launch_causal_tc(const DecodeArgs& a, int nqb, cudaStream_t s);

}  // namespace tq

struct tq_ctx {
  tq_config cfg;
  int device;
  tq::KindLayout kl, vl;
  tq::DeviceTables tab;
  void* dev_block;       // single allocation holding every device table
};

#endif  // TQ_INTERNAL_H_
