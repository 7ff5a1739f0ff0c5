// paged_gqa_decode + splitkv_combine for GB300 (sm_103a): the kernels and
// their launch templates. Each KV format's kernels are instantiated in a
// translation unit of its own (pa_decode_<format>.cu), so the formats
// compile in parallel; pa_decode.cu holds the host-side entry points.
//
// What is computed (heterogeneous C++ LLM engine article, section 4.3
// paged_attention_kernel; TFFInfer article, section 3.7.2 item 5 online
// softmax; Qwen2.5-7B engine article, section "3. GQA"): for sequence b and
// query head h with KV head j = h / g,
//   out[b][h] = sum_t softmax_t(q[b][h] . K_t * scale) V_t,  t < seq_len[b],
// where K_t / V_t live in slot t % bs of physical block block_table[b][t / bs]
// and quantised pools are read as (code - zp) * scale.
//
// Work decomposition (a GB300 design; the pages' sketch used one warp per
// head): a "unit" is one (sequence, kv head) pair and serves all g query
// heads of its group. The units are laid in (b, j) order on a cost line,
// each non-empty unit taking its pages plus a fixed number of phantom
// positions for its per-unit work; thread block i of G takes the slice
// [i*C/G, (i+1)*C/G) of that line and processes the real pages in it, so
// every SM gets the same share of work whatever the length mix. A unit that
// lies inside one slice is written straight to `out`; a unit cut by slice
// boundaries leaves one partial (o = acc / l, lse = m + log2 l) per slice,
// merged by the combine kernel with log-sum-exp weights.
//
// Inside a thread block: warp 0 is the producer. It sends each run's query
// rows by a bulk copy and issues the pages (K and V, plus the scales and
// zero points of quantised pools) into a ring of shared-memory stages by
// TMA, completing on mbarriers. Consumer warps take pages round-robin and
// keep a private online-softmax state per unit (fp32); at the end of a
// unit's run each deposits its state in a shared-memory stash, and a merger
// warp merges the deposited states and writes the row or the partial.
//
// Every wait is bounded: on expiry the thread block records
// PA_DEVERR_TIMEOUT, stops waiting and computing, keeps the barrier sequence
// (so no thread is stranded) and drains its outstanding copies before exit.
#pragma once

#include <float.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_kernels.h"
#include "pa_quant.cuh"

namespace pa {

namespace {

// Consumer warps per thread block. Four bf16 tensor-core warps (one per
// scheduler) keep up with HBM, so shared memory goes to the page ring; the
// uint8 tensor-core and the CUDA-core consumers are latency- or issue-bound
// and run eight.
template <int KV, bool TC, int BS>
constexpr int consumer_warps() {
  // Quantised tensor-core kernels run one block of 168-register threads per SM;
  // 12 warps (3 per sub-partition) still fit that budget. uint4 pages (32
  // tokens) measured faster with 8.
  return !TC ? 8 : (KV == PA_KV_BF16 ? 4 : (KV == PA_KV_UINT4 ? 8 : 10));
}
constexpr int kMaxSegs = 64;         // segments per window
constexpr int kMaxWinPages = 1024;   // pages per window (block-table entries staged in smem)
constexpr int kContPrev = 1, kContNext = 2;

// One contiguous run of pages of one unit inside a thread block's slice.
struct Seg {
  int32_t b, h;      // sequence, kv head
  int32_t lp0;       // first logical block of the run
  int32_t npages;    // pages in the run
  int32_t k0;        // index of the run's first page among the slice's pages
  int32_t len;       // sequence length (tokens)
  int32_t slot;      // partial slot (cta + unit), or -1 when written directly
  int32_t flags;     // kContPrev: continues the previous window's last run;
                     // kContNext: continues in the next window (no write yet)
  long long us;      // the unit's first position on the cost line
};

// Cost-balanced partition. The (sequence, kv head, block) work list is laid
// on a line where each non-empty unit occupies its pages followed by
// `unit_cost` phantom positions (the per-unit work: query load, state
// deposit and merge, partial write, expressed in pages); thread blocks take
// equal slices of that line and process the real pages in theirs. Blocks
// whose slice crosses many unit boundaries thus get fewer pages.
__device__ __forceinline__ int unit_span(int pages, int unit_cost) {
  return pages > 0 ? pages + unit_cost : 0;
}

template <int KV, int D, int BS>
struct PageGeom {
  static constexpr int kElemBits = KV == PA_KV_BF16 ? 16 : (KV == PA_KV_UINT4 ? 4 : 8);
  static constexpr int kPageBytes = BS * D * kElemBits / 8;      // one of K or V
  static constexpr int kMetaBytes = KV == PA_KV_BF16 ? 0 : D * 4;  // one of scale or zp
  static constexpr bool kHasZp = KV == PA_KV_UINT8 || KV == PA_KV_UINT4;  // fp8: scales only
  static constexpr int kStageBytes = 2 * kPageBytes + (kHasZp ? 4 : 2) * kMetaBytes;
  // offsets inside a stage (the zero-point offsets only where kHasZp)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kPageBytes;
  static constexpr int kOffKs = 2 * kPageBytes;
  static constexpr int kOffKz = kOffKs + kMetaBytes;
  static constexpr int kOffVs = kHasZp ? kOffKz + kMetaBytes : kOffKs + kMetaBytes;
  static constexpr int kOffVz = kOffVs + kMetaBytes;
};

template <int KV, int D, int BS, int G, int NS, int W, bool TC = false>
struct Smem {
  using PG = PageGeom<KV, D, BS>;
  static constexpr int kStages = W * NS;
  static constexpr int kQBytes = G * D * 2;
  // full[kStages], empty[kStages], qfull[2], qempty[2], deposited, merged, appended
  static constexpr size_t kOffBars = 0;
  static constexpr size_t kBarBytes = (2 * kStages + 7) * 8;
  static constexpr size_t kOffFlags = kBarBytes;  // int32 per stage
  static constexpr size_t kOffSegs = (kOffFlags + kStages * 4 + 15) / 16 * 16;
  static constexpr size_t kOffPlan = kOffSegs + kMaxSegs * sizeof(Seg);  // 32 int64
  static constexpr size_t kOffPhys = kOffPlan + 32 * 8;                   // int32 per window page
  static constexpr size_t kOffQ = (kOffPhys + kMaxWinPages * 4 + 127) / 128 * 128;
  static constexpr size_t kOffStash = kOffQ + 2 * kQBytes;
  static constexpr size_t kStashAccBytes = (size_t)W * G * D * 4;
  static constexpr size_t kOffStashML = kOffStash + kStashAccBytes;
  static constexpr size_t kOffPbuf = kOffStashML + W * G * 2 * 4;
  static constexpr size_t kPbufBytes = TC ? 0 : (size_t)W * BS * G * 4;  // CUDA-core consumer only
  static constexpr size_t kOffStages = (kOffPbuf + kPbufBytes + 1023) / 1024 * 1024;
  static constexpr size_t kBytes = kOffStages + (size_t)kStages * PG::kStageBytes + 1024;
};

struct DecodeParams {
  PoolMaps maps;
  PoolDev pool;
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* out;
  int32_t* pre_cost;             // [batch + 1] per-head cost-line prefix of the sequences
  float* part_o;
  float* part_lse;
  unsigned long long* tickets;  // per unit: (epoch << 24) | slices finished; 0 once merged
  unsigned long long epoch;     // 40-bit call tag, never 0
  int fused;                    // merge split units in this kernel (else: combine kernel)
  int early_plan;               // plan (reads of lengths / tables only) before waiting
                                // on the preceding kernel
  int batch;
  int num_q_heads;
  int group;
  int max_blocks;
  int unit_cost;                // phantom positions per unit on the cost line
  float scale_log2;
  // Several query tokens per sequence (kernels built with MQ): `batch`
  // counts virtual sequences v = b * n_cg + cg, column group cg of sequence
  // b, whose columns c are query token cg * tpg + c / g_heads and head
  // c % g_heads of the kv head's group; `group` is tpg * g_heads. q and out
  // are [B][n_q][Hq][D]. Single-token kernels: n_q = n_cg = tpg = 1,
  // g_heads = group.
  int n_q, n_cg, tpg, g_heads;
  // Fused decode step (single-token kernels): each sequence's last token,
  // row b of k_new / v_new (bf16 [batch][Hkv][D]), is stored into its block
  // (re-quantising it for quantised pools, as kv_quant_append does) by the
  // thread block that owns the unit's last page, before that page is read.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int append;
};

// The fused decode step's store for one unit: the new token (the last of
// `len`) of sequence b, kv head h, into its block, the record `page` (the
// unit's last page), K then V. Called by every consumer thread, kThreads of
// them (whole warps): lanes of a channel adjacent, channels in passes; warps
// whose channels are past head_dim sit a pass out. Not inlined: the page loop
// keeps its registers.
template <int KV, int BS>
__device__ __noinline__ void append_unit_tail(const PoolDev& pool, long long page, int b, int h, int len,
                                              const __nv_bfloat16* k_new, const __nv_bfloat16* v_new,
                                              int ct, int kThreads) {
  constexpr int TL = tok_lanes<BS>();
  const int D = pool.head_dim, Hkv = pool.num_kv_heads;
  const int lane = ct & 31, ts = lane & (TL - 1);
  const int old_cnt = (len - 1) % BS;                 // stored tokens before the new one
  const long long row0 = (long long)b - old_cnt;     // k_new row of slot s: row0 + s
  for (int base = 0; base < D; base += kThreads / TL) {
    const int c = base + ct / TL;
    if (base + (ct & ~31) / TL >= D) continue;        // the whole warp is past the last channel
#pragma unroll
    for (int is_v = 0; is_v < 2; ++is_v)
      append_block<KV, BS>(pool, page, is_v, c, ts, lane, old_cnt, old_cnt + 1, is_v ? v_new : k_new, row0,
                           Hkv, h);
  }
}

// ------------------------------------------------------------------ split-KV merge
//
// A unit cut by slice boundaries leaves one partial (o = acc / l,
// lse = m + log2 l) per slice. Merging them is the online-softmax update
// applied to whole states: M = max_s lse_s, w_s = 2^(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s. Slice i holds a partial of the unit (in
// slot i + u) iff its page range meets the unit's; slices between the first
// and last owner can be empty when there are more slices than pages.
//
// Cost-line arithmetic. Slice i of G is [T*i/G, T*(i+1)/G) of a line of T
// positions. When T*G < 2^32 (every launch short of billions of positions)
// the products and quotients are formed in 32-bit unsigned arithmetic: a
// 64-bit division is a long software sequence on the GPU, and these sit on
// the critical path of the planning before the first page is requested.
__device__ __forceinline__ bool line_small(long long T, long long G) {
  return T >= 0 && G > 0 && T <= 0xFFFFFFFFLL / G;
}
// first position of slice i (0 <= i <= G)
__device__ __forceinline__ long long slice_start(long long i, long long T, long long G, bool small) {
  return small ? (long long)((unsigned)T * (unsigned)i / (unsigned)G) : T * i / G;
}
// the slice containing position x (0 <= x < T)
__device__ __forceinline__ long long owner_of(long long x, long long T, long long G, bool small) {
  return small ? (long long)(((unsigned)x + 1u) * (unsigned)G - 1u) / (unsigned)T : ((x + 1) * G - 1) / T;
}

// Barrier among `threads` threads (whole warps) that all execute it with the
// same id; id 0 is the one __syncthreads uses.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

struct UnitSlices {
  long long first, last, us, n, T, G;
  bool small;  // line_small(T, G)
  __device__ __forceinline__ bool has_part(long long i) const {
    const long long a = slice_start(i, T, G, small), z = slice_start(i + 1, T, G, small);
    return (a > us ? a : us) < (z < us + n ? z : us + n);
  }
  __device__ __forceinline__ int count() const {
    int c = 0;
    for (long long i = first; i <= last; ++i) c += has_part(i);
    return c;
  }
};

// Merge the partials of unit u into out rows row0 .. row0+group-1, by threads
// tid = 0..nthr-1: a thread owns four channels of one head per column and
// up to kCols columns at a time, and folds the slices' (o, lse) pairs into a
// running (M, W, A) online; every load of a round (kCols columns x kBatch
// slices) is in flight at once. Partials are read through L2 (written by
// other thread blocks of this launch). Not inlined: the decode loop keeps
// its registers.
template <int D>
__device__ __noinline__ void merge_unit_partials(const UnitSlices& us, long long u, long long row0,
                                                 int group, const float* __restrict__ part_o,
                                                 const float* __restrict__ part_lse,
                                                 float* __restrict__ out, int tid, int nthr) {
  // four columns x two slices per round: a unit of 8 heads x 128 channels
  // (256 float4 columns) takes two rounds of loads on one warp
  constexpr int kBatch = 2, kCols = 4;
  const int ncol = group * D / 4;
  for (int c0 = tid; c0 < ncol; c0 += nthr * kCols) {
    float M[kCols], W[kCols], A[kCols][4];
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      M[j] = -INFINITY;
      W[j] = 0.0f;
      A[j][0] = A[j][1] = A[j][2] = A[j][3] = 0.0f;
    }
    for (long long i0 = us.first; i0 <= us.last; i0 += kBatch) {
      bool has[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) has[k] = i0 + k <= us.last && us.has_part(i0 + k);
      float l[kCols][kBatch];
      float4 o[kCols][kBatch];
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const int col = c0 + j * nthr;
        const int e0 = col * 4, h = e0 / D;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          l[j][k] = -INFINITY;
          o[j][k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (col < ncol && has[k]) {
            const long long slot = i0 + k + u;
            l[j][k] = __ldcg(part_lse + slot * group + h);
            o[j][k] = __ldcg(reinterpret_cast<const float4*>(part_o + slot * group * D + e0));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kCols; ++j)
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (l[j][k] == -INFINITY) continue;
          const float Mn = fmaxf(M[j], l[j][k]);
          const float a = M[j] == -INFINITY ? 0.0f : exp2f(M[j] - Mn), w = exp2f(l[j][k] - Mn);
          W[j] = W[j] * a + w;
          A[j][0] = A[j][0] * a + w * o[j][k].x;
          A[j][1] = A[j][1] * a + w * o[j][k].y;
          A[j][2] = A[j][2] * a + w * o[j][k].z;
          A[j][3] = A[j][3] * a + w * o[j][k].w;
          M[j] = Mn;
        }
    }
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int col = c0 + j * nthr;
      if (col >= ncol) continue;
      const float inv = W[j] > 0.0f ? 1.0f / W[j] : 0.0f;
      *reinterpret_cast<float4*>(out + row0 * D + col * 4) =
          make_float4(A[j][0] * inv, A[j][1] * inv, A[j][2] * inv, A[j][3] * inv);
    }
  }
}

// Sequence length clamped to what the table can hold; bad lengths count as 0.
__device__ __forceinline__ int seq_len_checked(const DecodeParams& p, int b, bool report) {
  const int len = p.seq_lens[b];
  if (len < 0 || (long long)len > (long long)p.max_blocks * p.pool.block_size) {
    if (report) set_error(p.pool.err, PA_DEVERR_SEQ_LEN);
    return 0;
  }
  return len;
}

// Virtual sequence v (see DecodeParams): its sequence, its length, its
// column count, the q / out row of its column c under kv head j, and the
// causal lag of its column 0 (query token i sees the tokens t < len -
// (n_q - 1 - i); the lag of column c is lag0 - c / g_heads).
template <bool MQ>
__device__ __forceinline__ int seq_of(const DecodeParams& p, int v) {
  return MQ ? v / p.n_cg : v;
}
template <bool MQ>
__device__ __forceinline__ int vlen_checked(const DecodeParams& p, int v, bool report) {
  return seq_len_checked(p, seq_of<MQ>(p, v), report);
}
template <bool MQ>
__device__ __forceinline__ int unit_cols(const DecodeParams& p, int v) {
  if constexpr (MQ) return min(p.tpg, p.n_q - (v % p.n_cg) * p.tpg) * p.g_heads;
  return p.group;
}
template <bool MQ>
__device__ __forceinline__ long long unit_row(const DecodeParams& p, int v, int j, int c) {
  if constexpr (MQ) {
    const int i = (v % p.n_cg) * p.tpg + c / p.g_heads;
    return ((long long)(v / p.n_cg) * p.n_q + i) * p.num_q_heads + (long long)j * p.g_heads + c % p.g_heads;
  }
  return (long long)v * p.num_q_heads + (long long)j * p.group + c;
}
template <bool MQ>
__device__ __forceinline__ int unit_lag0(const DecodeParams& p, int v) {
  return MQ ? p.n_q - 1 - (v % p.n_cg) * p.tpg : 0;
}


// Block-wide inclusive scan of one int per thread (all threads call).
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    const int t = warp_tot[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return x + before;
}

// ------------------------------------------------------------------ merge stash layout
//
// Each consumer warp deposits acc[h][c] of a unit into its stash rows, with
// the channel index XOR-swizzled so that the deposit's scattered stores hit
// 32 distinct banks: SWZ 0 keeps channel order (deposits of whole float4 /
// float2 per lane); SWZ 1 flips channel bits 3-4 by (h >> 1) (bf16 mma
// fragments: lanes differing in h >> 1 write the same column); SWZ 2 flips
// bits 0-1 by (h >> 1) (uint8 fragments, columns 4g + 2s); SWZ 3 also folds
// bit 5 into bit 2 (uint4 fragments, columns 8g + 2s). A lane's four (two)
// consecutive channels stay within one 16-byte (8-byte) word either way.
template <int SWZ>
__device__ __forceinline__ int stash_col(int h, int c) {
  if constexpr (SWZ == 0) return c;
  if constexpr (SWZ == 1) return c ^ (((h >> 1) & 3) << 3);
  if constexpr (SWZ == 2) return c ^ ((h >> 1) & 3);
  return c ^ ((h >> 1) & 3) ^ (((c >> 5) & 1) << 2);
}

// ------------------------------------------------------------------ consumer math (CUDA cores)
//
// Lane layout: lane l owns channels [l*CPL, (l+1)*CPL) of every row. Scores
// of a page are formed as per-lane partial dot products and reduced with a
// 5-step transpose butterfly over 32 (token, head) values at a time, after
// which lane l holds the score of head l % G and token (chunk*TOKC + l / G).
template <int KV, int D, int BS, int G>
struct FmaConsumer {
  static constexpr int CPL = D / 32;
  static constexpr int TOKC = 32 / G;
  static constexpr int NCH = BS / TOKC;
  static_assert(G * TOKC == 32 && NCH >= 1, "group padding");
  using PG = PageGeom<KV, D, BS>;

  float q[G][CPL];
  float acc[G][CPL];
  float m_run;  // for head lane % G
  float l_run;  // partial sum over this lane's tokens for head lane % G

  __device__ __forceinline__ void begin_unit(const uint16_t* q_smem, int g, float scale_log2) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float x = h < g ? __uint_as_float(((uint32_t)q_smem[h * D + lane * CPL + c]) << 16)
                              : 0.0f;
        q[h][c] = x * scale_log2;
        acc[h][c] = 0.0f;
      }
    }
    m_run = -INFINITY;
    l_run = 0.0f;
  }

  // Row t of a page (K or V) for this lane's channels, as floats.
  __device__ __forceinline__ void load_row(const uint8_t* page, const float* sc, const int32_t* zp,
                                           int t, float (&x)[CPL]) const {
    const int lane = threadIdx.x & 31;
    if (KV == PA_KV_BF16) {
      const uint16_t* row = reinterpret_cast<const uint16_t*>(page) + t * D + lane * CPL;
      if (CPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(row);
        x[0] = bf16_lo(w.x);
        x[1] = bf16_hi(w.x);
        x[2] = bf16_lo(w.y);
        x[3] = bf16_hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(row);
        x[0] = bf16_lo(w);
        x[1] = bf16_hi(w);
      }
    } else if (KV == PA_KV_FP8) {
      const uint8_t* row = page + t * D + lane * CPL;
      const uint32_t w = CPL == 4 ? *reinterpret_cast<const uint32_t*>(row)
                                  : (uint32_t) * reinterpret_cast<const uint16_t*>(row);
#pragma unroll
      for (int c = 0; c < CPL; ++c) x[c] = e4m3_to_float((w >> (8 * c)) & 0xFF) * sc[c];
    } else {
      uint32_t w;
      if (KV == PA_KV_UINT8) {
        const uint8_t* row = page + t * D + lane * CPL;
        w = CPL == 4 ? *reinterpret_cast<const uint32_t*>(row)
                     : (uint32_t) * reinterpret_cast<const uint16_t*>(row);
      } else {
        const uint8_t* row = page + t * (D / 2) + lane * CPL / 2;
        w = CPL == 4 ? (uint32_t) * reinterpret_cast<const uint16_t*>(row) : (uint32_t)*row;
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int code = KV == PA_KV_UINT8 ? (int)((w >> (8 * c)) & 0xFF) : (int)((w >> (4 * c)) & 0xF);
        x[c] = (float)(code - zp[c]) * sc[c];
      }
    }
  }

  template <bool MQ = false>
  __device__ __forceinline__ void page(const uint8_t* stage, int valid, float* pbuf, int to_end = 0) {
    const int lane = threadIdx.x & 31;
    // tokens this lane's column lane % G sees (several query tokens per
    // sequence: a causal lag; else the page's count)
    const int vc = MQ ? min(valid, to_end - lag_c) : valid;
    const uint8_t* kp = stage + PG::kOffK;
    const uint8_t* vp = stage + PG::kOffV;
    float ksc[CPL], vsc[CPL];
    int32_t kzp[CPL] = {}, vzp[CPL] = {};
    if (KV != PA_KV_BF16) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        ksc[c] = reinterpret_cast<const float*>(stage + PG::kOffKs)[lane * CPL + c];
        vsc[c] = reinterpret_cast<const float*>(stage + PG::kOffVs)[lane * CPL + c];
        if (PG::kHasZp) {
          kzp[c] = reinterpret_cast<const int32_t*>(stage + PG::kOffKz)[lane * CPL + c];
          vzp[c] = reinterpret_cast<const int32_t*>(stage + PG::kOffVz)[lane * CPL + c];
        }
      }
    }
    // ---- scores
    float s[NCH];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      float part[32];
#pragma unroll
      for (int tl = 0; tl < TOKC; ++tl) {
        const int t = ch * TOKC + tl;
        float kx[CPL];
        load_row(kp, ksc, kzp, t, kx);
#pragma unroll
        for (int c = 0; c < CPL; ++c) kx[c] = t < valid ? kx[c] : 0.0f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = 0.0f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) a = fmaf(q[h][c], kx[c], a);
          part[tl * G + h] = a;
        }
      }
#pragma unroll
      for (int off = 16, n = 16; off >= 1; off >>= 1, n >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
          const float send = upper ? part[i] : part[i + n];
          const float keep = upper ? part[i + n] : part[i];
          part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      const int t = ch * TOKC + lane / G;
      s[ch] = t < vc ? part[0] : -INFINITY;
    }
    // ---- online softmax (head lane % G)
    float pmax = s[0];
#pragma unroll
    for (int ch = 1; ch < NCH; ++ch) pmax = fmaxf(pmax, s[ch]);
#pragma unroll
    for (int off = G; off < 32; off <<= 1) pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, off));
    const float m_new = fmaxf(m_run, pmax);
    // a column that has seen no token yet keeps an empty state
    const float m_ref = MQ && m_new == -INFINITY ? 0.0f : m_new;
    const float alpha = exp2f(m_run - m_ref);
    float psum = 0.0f;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const float p = exp2f(s[ch] - m_ref);
      psum += p;
      pbuf[(ch * TOKC + lane / G) * G + lane % G] = p;
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    __syncwarp();
    // ---- P.V
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float a = __shfl_sync(0xffffffffu, alpha, h);
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[h][c] *= a;
    }
    for (int t = 0; t < valid; ++t) {
      float vx[CPL];
      load_row(vp, vsc, vzp, t, vx);
      float pt[G];
#pragma unroll
      for (int h = 0; h < G; ++h) pt[h] = pbuf[t * G + h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(pt[h], vx[c], acc[h][c]);
    }
    __syncwarp();
  }

  // Write this warp's state for the unit: m, l per head and acc[h][c].
  __device__ __forceinline__ void deposit(float* st_acc, float* st_ml) {
    const int lane = threadIdx.x & 31;
    float l = l_run;
#pragma unroll
    for (int off = G; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane < G) {
      st_ml[lane * 2] = m_run;
      st_ml[lane * 2 + 1] = l;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* dst = st_acc + h * D + lane * CPL;
      if constexpr (CPL == 4)
        *reinterpret_cast<float4*>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      else if constexpr (CPL == 2)
        *reinterpret_cast<float2*>(dst) = make_float2(acc[h][0], acc[h][1]);
      else
        for (int c = 0; c < CPL; ++c) dst[c] = acc[h][c];
    }
  }
  int lag_c = 0;  // causal lag of this lane's column lane % G
  // several query tokens per sequence: column c lags lag0 - c / gh tokens
  __device__ __forceinline__ void set_lags(int lag0, int gh) { lag_c = lag0 - (int)((threadIdx.x & 31) % G) / gh; }
  static constexpr int kStashSwz = 0;
};


// ------------------------------------------------------------------ consumer math (tensor cores)
//
// bf16 pools, page records staged by 2-D TMA with 128-byte swizzle: a record
// lands as [D/64 halves][BS K rows, then BS V rows][128 B], and 16-byte chunk
// c of row r sits at chunk c ^ (r % 8) of its 128-byte row, so ldmatrix reads
// are conflict-free.
//
// Scores of 16 tokens x the 8-wide head group come from mma.m16n8k16
// (A = K rows, B = Q^T held in registers for the whole unit, fp32
// accumulate). P.V uses A = V^T (ldmatrix.trans) and B = P^T, obtained from
// the score fragments with movmatrix.trans. P is split into a bf16 high part
// and a bf16 remainder (two mma per tile) so the weights keep ~16 bits.
// Lane t holds heads 2(t%4), 2(t%4)+1 throughout: the online-softmax state
// and the O^T accumulator columns line up without any exchange.
template <int D, int BS, int G>
struct MmaConsumerBf16 {
  static constexpr int KS = D / 16;   // k-steps of the score mma
  static constexpr int MT = D / 16;   // channel tiles of the P.V mma
  static constexpr int TT = BS / 16;  // 16-token tiles per page
  static constexpr int HALF_BYTES = BS * 128;   // one 64-channel half of K (or V)
  static constexpr int HALF_STRIDE = 2 * HALF_BYTES;  // a record half: K rows then V rows
  static_assert(G <= 8, "head group");

  uint32_t qf[KS][2];
  float o[MT][4];
  float m0, m1, l0, l1;
  float scale_log2;

  __device__ __forceinline__ void begin_unit(const uint16_t* q_smem, int g, float sl2) {
    const int lane = threadIdx.x & 31;
    const int h = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b0 = 0, b1 = 0;
      if (h < g) {
        b0 = *reinterpret_cast<const uint32_t*>(q_smem + h * D + ks * 16 + c2);
        b1 = *reinterpret_cast<const uint32_t*>(q_smem + h * D + ks * 16 + c2 + 8);
      }
      qf[ks][0] = b0;
      qf[ks][1] = b1;
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
    scale_log2 = sl2;
  }

  template <bool MQ = false>
  __device__ __forceinline__ void page(uint8_t* stage, int valid, float*, int to_end = 0) {
    const int lane = threadIdx.x & 31;
    const uint32_t kb = smem_u32(stage);
    const uint32_t vb = kb + HALF_BYTES;  // V rows follow K rows within each half
    // ---- scores S[token][head] for every 16-token tile
    float s[TT][4];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) s[tt][i] = 0.0f;
      const int row = tt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int chunk = (ks & 3) * 2 + (lane >> 4);  // 16-byte chunk within the 128-byte half-row
        const uint32_t addr = kb + (ks >> 2) * HALF_STRIDE + row * 128 + ((chunk ^ (row & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4(a, addr);
        mma_bf16_16816(s[tt], a, qf[ks][0], qf[ks][1]);
      }
    }
    // ---- online softmax for heads 2(t%4) and 2(t%4)+1
    const int tok = lane >> 2;
    // this lane's columns 2q, 2q+1 see the tokens below lim_a, lim_b (several query
    // tokens per sequence: causal lags; else both are the page's count)
    const int lim_a = MQ ? min(valid, to_end - lag_a) : valid, lim_b = MQ ? min(valid, to_end - lag_b) : valid;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const bool v0 = tt * 16 + tok < lim_a, v1 = tt * 16 + tok + 8 < lim_a;
      const bool w0 = tt * 16 + tok < lim_b, w1 = tt * 16 + tok + 8 < lim_b;
      s[tt][0] = v0 ? s[tt][0] * scale_log2 : -INFINITY;
      s[tt][1] = w0 ? s[tt][1] * scale_log2 : -INFINITY;
      s[tt][2] = v1 ? s[tt][2] * scale_log2 : -INFINITY;
      s[tt][3] = w1 ? s[tt][3] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[tt][0], s[tt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[tt][1], s[tt][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a column that has seen no token yet (several query tokens per
    // sequence) keeps an empty state instead of forming inf - inf
    const float r0 = MQ && n0 == -INFINITY ? 0.0f : n0, r1 = MQ && n1 == -INFINITY ? 0.0f : n1;
    const float a0 = ex2_approx(m0 - r0), a1 = ex2_approx(m1 - r1);
    m0 = n0;
    m1 = n1;
    uint32_t ph[TT][2], pl[TT][2];
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const float p0 = ex2_approx(s[tt][0] - r0), p1 = ex2_approx(s[tt][1] - r1);
      const float p2 = ex2_approx(s[tt][2] - r0), p3 = ex2_approx(s[tt][3] - r1);
      ps0 += p0 + p2;
      ps1 += p1 + p3;
      const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
      const uint32_t l01 = pack_bf16(p0 - bf16_lo_f(h01), p1 - bf16_hi_f(h01));
      const uint32_t l23 = pack_bf16(p2 - bf16_lo_f(h23), p3 - bf16_hi_f(h23));
      ph[tt][0] = movmatrix_trans(h01);
      ph[tt][1] = movmatrix_trans(h23);
      pl[tt][0] = movmatrix_trans(l01);
      pl[tt][1] = movmatrix_trans(l23);
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
    // ---- rows past the sequence end may hold anything: zero them so 0 * x
    // cannot turn into NaN inside the P.V mma
    if (valid < BS) {
      uint8_t* vrow = stage + HALF_BYTES;
      const int n16 = (BS - valid) * (D / 64) * 8;
      for (int i = lane; i < n16; i += 32) {
        const int half = i / ((BS - valid) * 8);
        const int rem = i % ((BS - valid) * 8);
        const int r = valid + rem / 8, c = rem % 8;
        *reinterpret_cast<uint4*>(vrow + half * HALF_STRIDE + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // ---- O^T[channel][head] += V^T[channel][token] P^T[token][head]
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const int j = lane >> 3;
      const int row = tt * 16 + (lane & 7) + (j >> 1) * 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int chunk = mt * 2 + (j & 1);  // 16-byte chunk across the 256-byte row
        const int half = chunk >> 3, c = chunk & 7;
        const uint32_t addr = vb + half * HALF_STRIDE + row * 128 + ((c ^ (row & 7)) << 4);
        uint32_t a[4];
        ldmatrix_x4_trans(a, addr);
        mma_bf16_16816(o[mt], a, ph[tt][0], ph[tt][1]);
        mma_bf16_16816(o[mt], a, pl[tt][0], pl[tt][1]);
      }
    }
    if (valid < BS) fence_proxy_async_smem();  // generic writes above, TMA writes next
  }

  __device__ __forceinline__ void deposit(float* st_acc, float* st_ml) {
    const int lane = threadIdx.x & 31;
    float s0 = l0, s1 = l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const int h0 = (lane & 3) * 2, ch = lane >> 2;
    if (lane < 4) {
      if (h0 < G) {
        st_ml[h0 * 2] = m0;
        st_ml[h0 * 2 + 1] = s0;
      }
      if (h0 + 1 < G) {
        st_ml[(h0 + 1) * 2] = m1;
        st_ml[(h0 + 1) * 2 + 1] = s1;
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if (h0 < G) {
        st_acc[h0 * D + stash_col<1>(h0, mt * 16 + ch)] = o[mt][0];
        st_acc[h0 * D + stash_col<1>(h0, mt * 16 + ch + 8)] = o[mt][2];
      }
      if (h0 + 1 < G) {
        st_acc[(h0 + 1) * D + stash_col<1>(h0 + 1, mt * 16 + ch)] = o[mt][1];
        st_acc[(h0 + 1) * D + stash_col<1>(h0 + 1, mt * 16 + ch + 8)] = o[mt][3];
      }
    }
  }
  int lag_a = 0, lag_b = 0;  // causal lags of this lane's columns 2q, 2q+1
  // several query tokens per sequence: column c lags lag0 - c / gh tokens
  __device__ __forceinline__ void set_lags(int lag0, int gh) {
    const int q = threadIdx.x & 3;
    lag_a = lag0 - (2 * q) / gh;
    lag_b = lag0 - (2 * q + 1) / gh;
  }
  static constexpr int kStashSwz = 1;
};


// ------------------------------------------------------------------ consumer math (tensor cores, uint8 KV)
//
// uint8 pools with head_dim 128: a page record (K codes, V codes, K scale,
// K zp, V scale, V zp) is staged by one 2-D TMA box with 128-byte swizzle
// (16-byte chunk c of 128-byte row r at chunk c ^ (r % 8)). With w_c = q_c * scale_c (per page and
// head) the score is s_t = sum_c w_c code_tc - sum_c w_c zp_c: the first sum
// is an f16 mma over exact integer codes (A = K codes, 16 tokens x 16
// channels per step; B = w, scaled by a power of two so its largest entry
// sits near 2^13, split into an f16 high part and an f16 remainder), the
// second an fp32 bias. Channel k-slots are permuted so that lane (g, q)
// reads channels 16k + 4q .. 16k + 4q + 3 of a row with one 32-bit load.
// P.V: raw[c][h] = sum_t code_tc p_th by an f16 mma (A = V codes^T gathered
// from four token rows, B = P^T via movmatrix, P split high + remainder),
// then o = alpha o + scale_c (raw - zp_c sum_t p_th) per page.
// Lane (g, q) holds heads 2q, 2q+1 of the online softmax and channels
// 32p + 4g .. 32p + 4g + 3 (p = 0..3) of the output.
template <int BS, int G>
struct MmaConsumerU8 {
  static constexpr int D = 128;
  static constexpr int KS = 8;        // 16-channel k-steps
  static constexpr int TT = BS / 16;  // 16-token tiles per page
  static constexpr int ROW = 128;     // bytes per token row
  static constexpr int PAGE = BS * ROW;
  static_assert(G <= 8, "head group");
  using PG = PageGeom<PA_KV_UINT8, 128, BS>;

  // Groups of up to 4 heads (one query token) split the per-page q*scale work:
  // lanes 16-31 prepare k-steps 4-7 of heads 0-3 and hand them to lanes 0-15
  // by shuffle; the mma's columns 4-7 then hold values no one stores.
  static constexpr bool kSplit = G <= 4;
  static constexpr int KH = kSplit ? KS / 2 : KS;  // k-steps of q*scale a lane prepares
  uint32_t qp[2 * KH];  // q[head] as bf16 pairs: channels 16k + 4q + {0,1} at 2k, {2,3} at 2k+1
  float o[8][4];    // O^T tile mt = 2p + s: rows -> channels 32p + 4g + 2s + {0, 1}
  float m0, m1, l0, l1;
  float scale_log2;

  __device__ __forceinline__ void begin_unit(const uint16_t* q_smem, int g, float sl2) {
    const int lane = threadIdx.x & 31;
    const int q4 = (lane & 3) * 4;
    const int hg = kSplit ? (lane >> 2) & 3 : lane >> 2;
    const int k0 = kSplit ? KH * (lane >> 4) : 0;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      uint2 w = make_uint2(0, 0);
      if (hg < g) w = *reinterpret_cast<const uint2*>(q_smem + hg * D + 16 * (k0 + k) + q4);
      qp[2 * k] = w.x;
      qp[2 * k + 1] = w.y;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
    scale_log2 = sl2;
  }

  // 16 bytes at byte offset `off` of the swizzled record (off 16-aligned)
  __device__ __forceinline__ static uint32_t sw(uint32_t base, uint32_t off) {
    const uint32_t r = off >> 7;
    return base + (r << 7) + ((((off >> 4) & 7) ^ (r & 7)) << 4);
  }
  __device__ __forceinline__ static float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
  }
  __device__ __forceinline__ static int4 lds_i4(uint32_t a) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
  }

  template <bool MQ = false>
  __device__ __forceinline__ void page(uint8_t* stage, int valid, float*, int to_end = 0) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    const uint32_t sb = smem_u32(stage);  // the whole record is swizzled
    // Swizzled addresses in closed form: the stage base is 1024-aligned and
    // each array starts on a known row phase (static_asserts below), so every
    // load is a per-lane base XOR a constant plus an immediate (checked
    // against the generic swizzle for all lanes).
    static_assert(PG::kOffK == 0 && PG::kOffV % 1024 == 0, "code rows start on an 8-row boundary");
    static_assert((PG::kOffKs / 128) % 8 == 0 && (PG::kOffKz / 128) % 8 == 4 &&
                      (PG::kOffVs / 128) % 8 == 0 && (PG::kOffVz / 128) % 8 == 4,
                  "metadata row phases");
    const uint32_t bq = sb + 16 * q;                 // K scales / zero points
    const uint32_t bg = sb + 16 * gq;                // V scales / zero points
    const uint32_t bk = sb + 144 * gq + 4 * q;       // K codes, row gq
    const uint32_t bv = sb + PG::kOffV + 288 * q + 16 * (gq >> 2) + 4 * (gq & 3);  // V codes, row 2q

    // ---- w = q * scale of this lane's head (its KH k-steps) and the head's
    // largest magnitude
    static_assert(!(kSplit && MQ), "several query tokens use groups of 8 columns");
    const uint32_t hx = kSplit ? 32u * (lane >> 4) : 0u, hoff = 8u * hx;  // k-steps 4-7: row phase + 2 rows
    float w[4 * KH];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const float4 sc = lds_f4(((bq ^ (16 * (k >> 1))) ^ hx) + hoff + PG::kOffKs + 128 * (k >> 1) + 64 * (k & 1));
      w[4 * k + 0] = bf16_lo(qp[2 * k]) * sc.x;
      w[4 * k + 1] = bf16_hi(qp[2 * k]) * sc.y;
      w[4 * k + 2] = bf16_lo(qp[2 * k + 1]) * sc.z;
      w[4 * k + 3] = bf16_hi(qp[2 * k + 1]) * sc.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(w[4 * k + j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if constexpr (kSplit) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
    int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    ex = ex < 1 ? 1 : ex;
    int sh = 140 - ex;  // 2^sh * amax lands in [2^13, 2^14)
    sh = sh < -120 ? -120 : (sh > 120 ? 120 : sh);
    const float f = __uint_as_float((uint32_t)(127 + sh) << 23);
    const float finv = __uint_as_float((uint32_t)(127 - sh) << 23);

    // ---- k-steps outermost: B = w * 2^sh split high + remainder (separate
    // accumulators keep the mma chains short), the zero-point bias, and the
    // score mma of every 16-token tile. Codes enter the mma as f16 subnormals
    // (a byte permuted against zero into a half's mantissa is code * 2^-24,
    // exactly), so the scores come out scaled by 2^-24.
    float sh_[TT][4], sl_[TT][4];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sh_[tt][i] = sl_[tt][i] = 0.0f;
    auto qk = [&](int k, uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        const uint32_t ka = (bk ^ (16 * k)) + tt * 16 * ROW;  // rows tt*16 + gq and + 8
        uint32_t c0, c1;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c0) : "r"(ka) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c1) : "r"(ka + 8 * ROW) : "memory");
        uint32_t a[4];
        a[0] = prmt(c0, 0u, 0x4140);
        a[1] = prmt(c1, 0u, 0x4140);
        a[2] = prmt(c0, 0u, 0x4342);
        a[3] = prmt(c1, 0u, 0x4342);
        mma_f16_16816(sh_[tt], a, bh0, bh1);
        mma_f16_16816(sl_[tt], a, bl0, bl1);
      }
    };
    float bias = 0.0f;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const int4 z = lds_i4(((bq ^ (16 * (k >> 1))) ^ hx) + hoff + PG::kOffKz + 128 * (k >> 1) + 64 * ((k & 1) ^ 1));
      const float w0 = w[4 * k] * f, w1 = w[4 * k + 1] * f, w2 = w[4 * k + 2] * f, w3 = w[4 * k + 3] * f;
      bias = fmaf(w0, (float)z.x, bias);
      bias = fmaf(w1, (float)z.y, bias);
      bias = fmaf(w2, (float)z.z, bias);
      bias = fmaf(w3, (float)z.w, bias);
      const uint32_t bh0 = pack_f16(w0, w1), bh1 = pack_f16(w2, w3);
      const float2 h01 = unpack_f16(bh0), h23 = unpack_f16(bh1);
      const uint32_t bl0 = pack_f16(w0 - h01.x, w1 - h01.y), bl1 = pack_f16(w2 - h23.x, w3 - h23.y);
      qk(k, bh0, bh1, bl0, bl1);
      if constexpr (kSplit)  // k-step k + 4, prepared by the lane 16 apart
        qk(k + KH, __shfl_xor_sync(0xffffffffu, bh0, 16), __shfl_xor_sync(0xffffffffu, bh1, 16),
           __shfl_xor_sync(0xffffffffu, bl0, 16), __shfl_xor_sync(0xffffffffu, bl1, 16));
    }
    if constexpr (kSplit) bias += __shfl_xor_sync(0xffffffffu, bias, 16);
    bias += __shfl_xor_sync(0xffffffffu, bias, 1);
    bias += __shfl_xor_sync(0xffffffffu, bias, 2);
    // heads 2q, 2q+1 of the score fragments: bias and scale from their lanes
    const float bias0 = __shfl_sync(0xffffffffu, bias, 8 * q);
    const float bias1 = __shfl_sync(0xffffffffu, bias, 8 * q + 4);
    const float mul0 = __shfl_sync(0xffffffffu, finv, 8 * q) * scale_log2;
    const float mul1 = __shfl_sync(0xffffffffu, finv, 8 * q + 4) * scale_log2;
    float s[TT][4];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[tt][i] = sh_[tt][i] + sl_[tt][i];
    // ---- online softmax for heads 2q, 2q+1
    // this lane's columns 2q, 2q+1 see the tokens below lim_a, lim_b (several query
    // tokens per sequence: causal lags; else both are the page's count)
    const int lim_a = MQ ? min(valid, to_end - lag_a) : valid, lim_b = MQ ? min(valid, to_end - lag_b) : valid;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const bool v0 = tt * 16 + gq < lim_a, v1 = tt * 16 + gq + 8 < lim_a;
      const bool w0 = tt * 16 + gq < lim_b, w1 = tt * 16 + gq + 8 < lim_b;
      s[tt][0] = v0 ? fmaf(s[tt][0], 0x1p24f, -bias0) * mul0 : -INFINITY;
      s[tt][1] = w0 ? fmaf(s[tt][1], 0x1p24f, -bias1) * mul1 : -INFINITY;
      s[tt][2] = v1 ? fmaf(s[tt][2], 0x1p24f, -bias0) * mul0 : -INFINITY;
      s[tt][3] = w1 ? fmaf(s[tt][3], 0x1p24f, -bias1) * mul1 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[tt][0], s[tt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[tt][1], s[tt][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a column that has seen no token yet (several query tokens per
    // sequence) keeps an empty state instead of forming inf - inf
    const float r0 = MQ && n0 == -INFINITY ? 0.0f : n0, r1 = MQ && n1 == -INFINITY ? 0.0f : n1;
    const float a0 = ex2_approx(m0 - r0), a1 = ex2_approx(m1 - r1);
    m0 = n0;
    m1 = n1;
    uint32_t ph[TT][2], pl[TT][2];
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const float p0 = ex2_approx(s[tt][0] - r0), p1 = ex2_approx(s[tt][1] - r1);
      const float p2 = ex2_approx(s[tt][2] - r0), p3 = ex2_approx(s[tt][3] - r1);
      ps0 += p0 + p2;
      ps1 += p1 + p3;
      const uint32_t h01 = pack_f16(p0, p1), h23 = pack_f16(p2, p3);
      const float2 f01 = unpack_f16(h01), f23 = unpack_f16(h23);
      ph[tt][0] = movmatrix_trans(h01);
      ph[tt][1] = movmatrix_trans(h23);
      pl[tt][0] = movmatrix_trans(pack_f16(p0 - f01.x, p1 - f01.y));
      pl[tt][1] = movmatrix_trans(pack_f16(p2 - f23.x, p3 - f23.y));
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
    // page sums of p per head (for the zero-point term of the fold)
    float sum0 = ps0, sum1 = ps1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, off);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, off);
    }
    // ---- raw[c][h] = sum_t code_tc p_th; codes past the sequence end are
    // finite integers met by p = 0, so they add nothing. The codes are f16
    // subnormals (code * 2^-24) here too: o accumulates in units of 2^-24
    // (zp sum_p scaled to match) and is scaled back when deposited.
    sum0 *= 0x1p-24f;
    sum1 *= 0x1p-24f;
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      float raw0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, raw1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint32_t va = bv ^ (32 * pr), vo = va ^ 16;  // rows 2q (+8) and 2q + 1 (+8)
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        uint32_t W0, W1, W2, W3;  // tokens tt*16 + 2q + {0, 1, 8, 9}
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W0) : "r"(va + tt * 16 * ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W1) : "r"(vo + tt * 16 * ROW + ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W2) : "r"(va + tt * 16 * ROW + 8 * ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W3) : "r"(vo + tt * 16 * ROW + 9 * ROW) : "memory");
        const uint32_t u01 = prmt(W0, W1, 0x5140), u23 = prmt(W0, W1, 0x7362);
        const uint32_t v01 = prmt(W2, W3, 0x5140), v23 = prmt(W2, W3, 0x7362);
        uint32_t A0[4], A1[4];
        A0[0] = prmt(u01, 0u, 0x4140);  // channel +0, tokens t0 t1
        A0[1] = prmt(u01, 0u, 0x4342);  // channel +1
        A0[2] = prmt(v01, 0u, 0x4140);  // channel +0, tokens t2 t3
        A0[3] = prmt(v01, 0u, 0x4342);
        A1[0] = prmt(u23, 0u, 0x4140);  // channel +2
        A1[1] = prmt(u23, 0u, 0x4342);  // channel +3
        A1[2] = prmt(v23, 0u, 0x4140);
        A1[3] = prmt(v23, 0u, 0x4342);
        mma_f16_16816(raw0, A0, ph[tt][0], ph[tt][1]);
        mma_f16_16816(raw0, A0, pl[tt][0], pl[tt][1]);
        mma_f16_16816(raw1, A1, ph[tt][0], ph[tt][1]);
        mma_f16_16816(raw1, A1, pl[tt][0], pl[tt][1]);
      }
      // fold: o = alpha o + scale (raw - zp * sum_p)
      const float4 sc = lds_f4((bg ^ (16 * pr)) + PG::kOffVs + 128 * pr);  // channels 32pr + 4gq .. + 3
      const int4 z = lds_i4((bg ^ (16 * (4 ^ pr))) + PG::kOffVz + 128 * pr);
      float* oa = o[2 * pr];
      float* ob = o[2 * pr + 1];
      oa[0] = fmaf(a0, oa[0], sc.x * fmaf(-(float)z.x, sum0, raw0[0]));
      oa[1] = fmaf(a1, oa[1], sc.x * fmaf(-(float)z.x, sum1, raw0[1]));
      oa[2] = fmaf(a0, oa[2], sc.y * fmaf(-(float)z.y, sum0, raw0[2]));
      oa[3] = fmaf(a1, oa[3], sc.y * fmaf(-(float)z.y, sum1, raw0[3]));
      ob[0] = fmaf(a0, ob[0], sc.z * fmaf(-(float)z.z, sum0, raw1[0]));
      ob[1] = fmaf(a1, ob[1], sc.z * fmaf(-(float)z.z, sum1, raw1[1]));
      ob[2] = fmaf(a0, ob[2], sc.w * fmaf(-(float)z.w, sum0, raw1[2]));
      ob[3] = fmaf(a1, ob[3], sc.w * fmaf(-(float)z.w, sum1, raw1[3]));
    }
  }

  __device__ __forceinline__ void deposit(float* st_acc, float* st_ml) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    float s0 = l0, s1 = l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const int h0 = 2 * q;
    if (lane < 4) {
      if (h0 < G) {
        st_ml[h0 * 2] = m0;
        st_ml[h0 * 2 + 1] = s0;
      }
      if (h0 + 1 < G) {
        st_ml[(h0 + 1) * 2] = m1;
        st_ml[(h0 + 1) * 2 + 1] = s1;
      }
    }
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
#pragma unroll
      for (int sd = 0; sd < 2; ++sd) {
        const int c = 32 * pr + 4 * gq + 2 * sd;
        const float* ot = o[2 * pr + sd];
        if (h0 < G) {  // o is held in units of 2^-24
          st_acc[h0 * D + stash_col<2>(h0, c)] = ot[0] * 0x1p24f;
          st_acc[h0 * D + stash_col<2>(h0, c + 1)] = ot[2] * 0x1p24f;
        }
        if (h0 + 1 < G) {
          st_acc[(h0 + 1) * D + stash_col<2>(h0 + 1, c)] = ot[1] * 0x1p24f;
          st_acc[(h0 + 1) * D + stash_col<2>(h0 + 1, c + 1)] = ot[3] * 0x1p24f;
        }
      }
    }
  }
  int lag_a = 0, lag_b = 0;  // causal lags of this lane's columns 2q, 2q+1
  // several query tokens per sequence: column c lags lag0 - c / gh tokens
  __device__ __forceinline__ void set_lags(int lag0, int gh) {
    const int q = threadIdx.x & 3;
    lag_a = lag0 - (2 * q) / gh;
    lag_b = lag0 - (2 * q + 1) / gh;
  }
  static constexpr int kStashSwz = 2;
};


// ------------------------------------------------------------------ consumer math (tensor cores, fp8 KV)
//
// fp8 (E4M3) pools with head_dim 128: a record (K codes, V codes, K scale,
// V scale) is staged like a uint8 record, one 2-D TMA box with 128-byte
// swizzle. The uint8 scheme without zero points: every E4M3 value is an f16
// value (3 mantissa bits, magnitudes 2^-9 .. 448), so the hardware
// conversion feeds exact values to the same f16 mma. Scores:
// s_t = sum_c w_c value_tc with w_c = q_c * scale_c scaled by a power of two
// and split into an f16 high part and remainder. P.V: raw[c][h] =
// sum_t value_tc p_th, then o = alpha o + scale_c raw per page. A slot past
// the sequence end may hold any bit pattern, NaN included, which p = 0
// would not cancel: its codes are replaced by zero before P.V.
template <int BS, int G>
struct MmaConsumerFp8 {
  static constexpr int D = 128;
  static constexpr int KS = 8;        // 16-channel k-steps
  static constexpr int TT = BS / 16;  // 16-token tiles per page
  static constexpr int ROW = 128;     // bytes per token row
  static_assert(G <= 8, "head group");
  using PG = PageGeom<PA_KV_FP8, 128, BS>;

  // Groups of up to 4 heads (one query token) split the per-page q*scale work
  // as in the uint8 consumer: lanes 16-31 prepare k-steps 4-7 of heads 0-3.
  static constexpr bool kSplit = G <= 4;
  static constexpr int KH = kSplit ? KS / 2 : KS;  // k-steps of q*scale a lane prepares
  uint32_t qp[2 * KH];  // q[head] as bf16 pairs: channels 16k + 4q + {0,1} at 2k, {2,3} at 2k+1
  float o[8][4];    // O^T tile mt = 2p + s: rows -> channels 32p + 4g + 2s + {0, 1}
  float m0, m1, l0, l1;
  float scale_log2;

  __device__ __forceinline__ void begin_unit(const uint16_t* q_smem, int g, float sl2) {
    const int lane = threadIdx.x & 31;
    const int q4 = (lane & 3) * 4;
    const int hg = kSplit ? (lane >> 2) & 3 : lane >> 2;
    const int k0 = kSplit ? KH * (lane >> 4) : 0;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      uint2 w = make_uint2(0, 0);
      if (hg < g) w = *reinterpret_cast<const uint2*>(q_smem + hg * D + 16 * (k0 + k) + q4);
      qp[2 * k] = w.x;
      qp[2 * k + 1] = w.y;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
    scale_log2 = sl2;
  }

  __device__ __forceinline__ static float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
  }

  template <bool MQ = false>
  __device__ __forceinline__ void page(uint8_t* stage, int valid, float*, int to_end = 0) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    const uint32_t sb = smem_u32(stage);  // the whole record is swizzled
    // Swizzled addresses in closed form, as in the uint8 consumer: the stage
    // base is 1024-aligned and the K scales start on row phase 0, the V
    // scales on row phase 4 (no zero points between them).
    static_assert(PG::kOffK == 0 && PG::kOffV % 1024 == 0, "code rows start on an 8-row boundary");
    static_assert((PG::kOffKs / 128) % 8 == 0 && (PG::kOffVs / 128) % 8 == 4, "metadata row phases");
    static_assert(PG::kStageBytes % 1024 == 0, "every stage base stays 1024-aligned");
    const uint32_t bq = sb + 16 * q;                 // K scales
    const uint32_t bg = sb + 16 * gq;                // V scales
    const uint32_t bk = sb + 144 * gq + 4 * q;       // K codes, row gq
    const uint32_t bv = sb + PG::kOffV + 288 * q + 16 * (gq >> 2) + 4 * (gq & 3);  // V codes, row 2q

    // ---- w = q * scale of this lane's head (its KH k-steps) and the head's
    // largest magnitude
    static_assert(!(kSplit && MQ), "several query tokens use groups of 8 columns");
    const uint32_t hx = kSplit ? 32u * (lane >> 4) : 0u, hoff = 8u * hx;  // k-steps 4-7: row phase + 2 rows
    float w[4 * KH];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const float4 sc = lds_f4(((bq ^ (16 * (k >> 1))) ^ hx) + hoff + PG::kOffKs + 128 * (k >> 1) + 64 * (k & 1));
      w[4 * k + 0] = bf16_lo(qp[2 * k]) * sc.x;
      w[4 * k + 1] = bf16_hi(qp[2 * k]) * sc.y;
      w[4 * k + 2] = bf16_lo(qp[2 * k + 1]) * sc.z;
      w[4 * k + 3] = bf16_hi(qp[2 * k + 1]) * sc.w;
#pragma unroll
      for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(w[4 * k + j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if constexpr (kSplit) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
    int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    ex = ex < 1 ? 1 : ex;
    int sh = 140 - ex;  // 2^sh * amax lands in [2^13, 2^14)
    sh = sh < -120 ? -120 : (sh > 120 ? 120 : sh);
    const float f = __uint_as_float((uint32_t)(127 + sh) << 23);
    const float finv = __uint_as_float((uint32_t)(127 - sh) << 23);

    // ---- k-steps outermost: B = w * 2^sh split high + remainder, and the
    // score mma of every 16-token tile
    float sh_[TT][4], sl_[TT][4];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sh_[tt][i] = sl_[tt][i] = 0.0f;
    auto qk = [&](int k, uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        const uint32_t ka = (bk ^ (16 * k)) + tt * 16 * ROW;  // rows tt*16 + gq and + 8
        uint32_t c0, c1;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c0) : "r"(ka) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(c1) : "r"(ka + 8 * ROW) : "memory");
        uint32_t a[4];
        a[0] = e4m3x2_lo_to_f16x2(c0);  // channels 16k + 4q + {0, 1}
        a[1] = e4m3x2_lo_to_f16x2(c1);
        a[2] = e4m3x2_hi_to_f16x2(c0);  // channels 16k + 4q + {2, 3}
        a[3] = e4m3x2_hi_to_f16x2(c1);
        mma_f16_16816(sh_[tt], a, bh0, bh1);
        mma_f16_16816(sl_[tt], a, bl0, bl1);
      }
    };
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const float w0 = w[4 * k] * f, w1 = w[4 * k + 1] * f, w2 = w[4 * k + 2] * f, w3 = w[4 * k + 3] * f;
      const uint32_t bh0 = pack_f16(w0, w1), bh1 = pack_f16(w2, w3);
      const float2 h01 = unpack_f16(bh0), h23 = unpack_f16(bh1);
      const uint32_t bl0 = pack_f16(w0 - h01.x, w1 - h01.y), bl1 = pack_f16(w2 - h23.x, w3 - h23.y);
      qk(k, bh0, bh1, bl0, bl1);
      if constexpr (kSplit)  // k-step k + 4, prepared by the lane 16 apart
        qk(k + KH, __shfl_xor_sync(0xffffffffu, bh0, 16), __shfl_xor_sync(0xffffffffu, bh1, 16),
           __shfl_xor_sync(0xffffffffu, bl0, 16), __shfl_xor_sync(0xffffffffu, bl1, 16));
    }
    // heads 2q, 2q+1 of the score fragments: the scale from their lanes
    const float mul0 = __shfl_sync(0xffffffffu, finv, 8 * q) * scale_log2;
    const float mul1 = __shfl_sync(0xffffffffu, finv, 8 * q + 4) * scale_log2;
    // ---- online softmax for heads 2q, 2q+1 (rows past the end selected out)
    float s[TT][4];
    // this lane's columns 2q, 2q+1 see the tokens below lim_a, lim_b (several query
    // tokens per sequence: causal lags; else both are the page's count)
    const int lim_a = MQ ? min(valid, to_end - lag_a) : valid, lim_b = MQ ? min(valid, to_end - lag_b) : valid;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const bool v0 = tt * 16 + gq < lim_a, v1 = tt * 16 + gq + 8 < lim_a;
      const bool w0 = tt * 16 + gq < lim_b, w1 = tt * 16 + gq + 8 < lim_b;
      s[tt][0] = v0 ? (sh_[tt][0] + sl_[tt][0]) * mul0 : -INFINITY;
      s[tt][1] = w0 ? (sh_[tt][1] + sl_[tt][1]) * mul1 : -INFINITY;
      s[tt][2] = v1 ? (sh_[tt][2] + sl_[tt][2]) * mul0 : -INFINITY;
      s[tt][3] = w1 ? (sh_[tt][3] + sl_[tt][3]) * mul1 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[tt][0], s[tt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[tt][1], s[tt][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a column that has seen no token yet (several query tokens per
    // sequence) keeps an empty state instead of forming inf - inf
    const float r0 = MQ && n0 == -INFINITY ? 0.0f : n0, r1 = MQ && n1 == -INFINITY ? 0.0f : n1;
    const float a0 = ex2_approx(m0 - r0), a1 = ex2_approx(m1 - r1);
    m0 = n0;
    m1 = n1;
    uint32_t ph[TT][2], pl[TT][2];
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const float p0 = ex2_approx(s[tt][0] - r0), p1 = ex2_approx(s[tt][1] - r1);
      const float p2 = ex2_approx(s[tt][2] - r0), p3 = ex2_approx(s[tt][3] - r1);
      ps0 += p0 + p2;
      ps1 += p1 + p3;
      const uint32_t h01 = pack_f16(p0, p1), h23 = pack_f16(p2, p3);
      const float2 f01 = unpack_f16(h01), f23 = unpack_f16(h23);
      ph[tt][0] = movmatrix_trans(h01);
      ph[tt][1] = movmatrix_trans(h23);
      pl[tt][0] = movmatrix_trans(pack_f16(p0 - f01.x, p1 - f01.y));
      pl[tt][1] = movmatrix_trans(pack_f16(p2 - f23.x, p3 - f23.y));
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
    // ---- raw[c][h] = sum_t value_tc p_th
    const bool tail = valid < BS;  // warp-uniform
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      float raw0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, raw1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint32_t va = bv ^ (32 * pr), vo = va ^ 16;  // rows 2q (+8) and 2q + 1 (+8)
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        uint32_t W0, W1, W2, W3;  // tokens tt*16 + 2q + {0, 1, 8, 9}
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W0) : "r"(va + tt * 16 * ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W1) : "r"(vo + tt * 16 * ROW + ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W2) : "r"(va + tt * 16 * ROW + 8 * ROW) : "memory");
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(W3) : "r"(vo + tt * 16 * ROW + 9 * ROW) : "memory");
        if (tail) {
          const int t0 = tt * 16 + 2 * q;
          W0 = t0 < valid ? W0 : 0u;
          W1 = t0 + 1 < valid ? W1 : 0u;
          W2 = t0 + 8 < valid ? W2 : 0u;
          W3 = t0 + 9 < valid ? W3 : 0u;
        }
        const uint32_t u01 = prmt(W0, W1, 0x5140), u23 = prmt(W0, W1, 0x7362);
        const uint32_t v01 = prmt(W2, W3, 0x5140), v23 = prmt(W2, W3, 0x7362);
        uint32_t A0[4], A1[4];
        A0[0] = e4m3x2_lo_to_f16x2(u01);  // channel +0, tokens t0 t1
        A0[1] = e4m3x2_hi_to_f16x2(u01);  // channel +1
        A0[2] = e4m3x2_lo_to_f16x2(v01);  // channel +0, tokens t2 t3
        A0[3] = e4m3x2_hi_to_f16x2(v01);
        A1[0] = e4m3x2_lo_to_f16x2(u23);  // channel +2
        A1[1] = e4m3x2_hi_to_f16x2(u23);  // channel +3
        A1[2] = e4m3x2_lo_to_f16x2(v23);
        A1[3] = e4m3x2_hi_to_f16x2(v23);
        mma_f16_16816(raw0, A0, ph[tt][0], ph[tt][1]);
        mma_f16_16816(raw0, A0, pl[tt][0], pl[tt][1]);
        mma_f16_16816(raw1, A1, ph[tt][0], ph[tt][1]);
        mma_f16_16816(raw1, A1, pl[tt][0], pl[tt][1]);
      }
      // fold: o = alpha o + scale raw (V scales on row phase 4)
      const float4 sc = lds_f4((bg ^ (16 * (4 ^ pr))) + PG::kOffVs + 128 * pr);  // channels 32pr + 4gq ..
      float* oa = o[2 * pr];
      float* ob = o[2 * pr + 1];
      oa[0] = fmaf(a0, oa[0], sc.x * raw0[0]);
      oa[1] = fmaf(a1, oa[1], sc.x * raw0[1]);
      oa[2] = fmaf(a0, oa[2], sc.y * raw0[2]);
      oa[3] = fmaf(a1, oa[3], sc.y * raw0[3]);
      ob[0] = fmaf(a0, ob[0], sc.z * raw1[0]);
      ob[1] = fmaf(a1, ob[1], sc.z * raw1[1]);
      ob[2] = fmaf(a0, ob[2], sc.w * raw1[2]);
      ob[3] = fmaf(a1, ob[3], sc.w * raw1[3]);
    }
  }

  __device__ __forceinline__ void deposit(float* st_acc, float* st_ml) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    float s0 = l0, s1 = l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const int h0 = 2 * q;
    if (lane < 4) {
      if (h0 < G) {
        st_ml[h0 * 2] = m0;
        st_ml[h0 * 2 + 1] = s0;
      }
      if (h0 + 1 < G) {
        st_ml[(h0 + 1) * 2] = m1;
        st_ml[(h0 + 1) * 2 + 1] = s1;
      }
    }
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
#pragma unroll
      for (int sd = 0; sd < 2; ++sd) {
        const int c = 32 * pr + 4 * gq + 2 * sd;
        const float* ot = o[2 * pr + sd];
        if (h0 < G) {
          st_acc[h0 * D + stash_col<2>(h0, c)] = ot[0];
          st_acc[h0 * D + stash_col<2>(h0, c + 1)] = ot[2];
        }
        if (h0 + 1 < G) {
          st_acc[(h0 + 1) * D + stash_col<2>(h0 + 1, c)] = ot[1];
          st_acc[(h0 + 1) * D + stash_col<2>(h0 + 1, c + 1)] = ot[3];
        }
      }
    }
  }
  int lag_a = 0, lag_b = 0;  // causal lags of this lane's columns 2q, 2q+1
  // several query tokens per sequence: column c lags lag0 - c / gh tokens
  __device__ __forceinline__ void set_lags(int lag0, int gh) {
    const int q = threadIdx.x & 3;
    lag_a = lag0 - (2 * q) / gh;
    lag_b = lag0 - (2 * q + 1) / gh;
  }
  static constexpr int kStashSwz = 2;
};


// ------------------------------------------------------------------ consumer math (tensor cores, uint4 KV)
//
// Packed uint4 pools with head_dim 128: like the uint8 consumer, on a page
// record of 64-byte token rows (two per 128-byte swizzled row). A 32-bit load
// of a token row carries 8 channels as nibbles (channel 2i low, 2i+1 high);
// masking gives the even channels, a shift the odd ones, each as bytes that
// become exact f16 integers. Scores: lane (g, q) loads bytes 16k + 4q of a
// row = channels 32k + 8q .. +7 and feeds two k-steps with them (even
// channels in the first B/A slots, odd in the second); B = w for the same
// channels. P.V: lane (g, q) owns channels 64o + 8g + 2s + {0, 1} of the
// O^T tiles 4o + s and gathers them from four token rows.
template <int BS, int G>
struct MmaConsumerU4 {
  static constexpr int D = 128;
  static constexpr int TT = BS / 16;
  static constexpr int ROWB = 64;  // bytes per token row
  static_assert(G <= 8, "head group");
  using PG = PageGeom<PA_KV_UINT4, 128, BS>;

  // Groups of up to 4 heads (one query token) split the per-page q*scale work:
  // lanes 16-31 prepare k-steps 2 and 3 of heads 0-3 and hand them to lanes
  // 0-15 by shuffle; the mma's columns 4-7 then hold values no one stores.
  static constexpr bool kSplit = G <= 4;
  static constexpr int KH = kSplit ? 2 : 4;  // k-steps of q*scale a lane prepares
  uint32_t qp[4 * KH];  // q[head] bf16 pairs, channels 32k + 8q + {0,1},{2,3},{4,5},{6,7} at 4k..4k+3
  float o[8][4];    // O^T tile mt = 4o + s: rows -> channels 64o + 8g + 2s + {0, 1}
  float m0, m1, l0, l1;
  float scale_log2;

  __device__ __forceinline__ static uint32_t sw(uint32_t base, uint32_t off) {
    const uint32_t r = off >> 7;
    return base + (r << 7) + ((((off >> 4) & 7) ^ (r & 7)) << 4) + (off & 15);
  }
  __device__ __forceinline__ static uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
  }
  __device__ __forceinline__ static float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
  }
  __device__ __forceinline__ static int4 lds_i4(uint32_t a) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
  }

  __device__ __forceinline__ void begin_unit(const uint16_t* q_smem, int g, float sl2) {
    const int lane = threadIdx.x & 31;
    const int q8 = (lane & 3) * 8;
    // groups of up to 4 heads: lanes 16-31 hold k-steps 2, 3 of heads 0-3
    const int hg = kSplit ? (lane >> 2) & 3 : lane >> 2;
    const int k0 = kSplit ? 2 * (lane >> 4) : 0;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (hg < g) w = *reinterpret_cast<const uint4*>(q_smem + hg * D + 32 * (k0 + k) + q8);
      qp[4 * k] = w.x;
      qp[4 * k + 1] = w.y;
      qp[4 * k + 2] = w.z;
      qp[4 * k + 3] = w.w;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][i] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
    scale_log2 = sl2;
  }

  template <bool MQ = false>
  __device__ __forceinline__ void page(uint8_t* stage, int valid, float*, int to_end = 0) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    const uint32_t sb = smem_u32(stage);  // the whole record is swizzled
    // Swizzled addresses in closed form (a per-lane base XOR a constant plus
    // an immediate; the stage base is 1024-aligned and each array starts on
    // a known row phase), checked against the generic swizzle for all lanes.
    static_assert(PG::kOffK == 0 && PG::kOffV % 1024 == 0, "code rows start on an 8-row boundary");
    static_assert((PG::kOffKs / 128) % 8 == 0 && (PG::kOffKz / 128) % 8 == 4 &&
                      (PG::kOffVs / 128) % 8 == 0 && (PG::kOffVz / 128) % 8 == 4,
                  "metadata row phases");
    const uint32_t bq = sb + 32 * q;  // K scales / zero points
    const uint32_t bkc = sb + 128 * (gq >> 1) + 64 * (gq & 1) + 16 * (gq >> 1) + 4 * q;  // K codes, row gq
    const uint32_t bvc = sb + PG::kOffV + 128 * q + 16 * ((gq >> 2) ^ q) + 4 * (gq & 3);  // V codes, row 2q
    const uint32_t bvm = sb + 128 * (gq >> 2) + 32 * (gq & 3) + 16 * (gq >> 2);  // V scales / zero points

    // ---- w = q * scale of this lane's head (channels 32k + 8q + j of its KH
    // k-steps) and the head's largest magnitude
    static_assert(!(kSplit && MQ), "several query tokens use groups of 8 columns");
    const uint32_t hx = kSplit ? 32u * (lane >> 4) : 0u, hoff = 8u * hx;  // k-steps 2, 3: row phase + 2 rows
    float w[8 * KH];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const uint32_t ks = ((bq ^ (32 * (k >> 1))) ^ hx) + hoff + PG::kOffKs + 128 * k;
      const float4 s0 = lds_f4(ks + 16 * (k & 1));
      const float4 s1 = lds_f4(ks + 16 * ((k & 1) ^ 1));
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t pr = qp[4 * k + j / 2];
        w[8 * k + j] = ((j & 1) ? bf16_hi(pr) : bf16_lo(pr)) * sc[j];
        amax = fmaxf(amax, fabsf(w[8 * k + j]));
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if constexpr (kSplit) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
    int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    ex = ex < 1 ? 1 : ex;
    int sh = 140 - ex;
    sh = sh < -120 ? -120 : (sh > 120 ? 120 : sh);
    const float f = __uint_as_float((uint32_t)(127 + sh) << 23);
    const float finv = __uint_as_float((uint32_t)(127 - sh) << 23);

    // Codes enter the mma as f16 subnormals: masking a nibble into a half's low
    // mantissa bits, exponent zero, gives code * 2^-24 (bits 0-3) or code * 2^-20
    // (bits 4-7) exactly, with no conversion. The 2^-20 channels (odd j) take
    // q*scale*f / 16, so every product is code * q*scale*f * 2^-24; the 2^24
    // comes back in the score below. Channel pairs per k-step: (j0, j4) | (j1, j5),
    // then (j2, j6) | (j3, j7), as the masks of a code word and of its 8-bit shift
    // deliver them.
    const float f16th = f * 0.0625f;
    float sh_[TT][4], sl_[TT][4];
#pragma unroll
    for (int tt = 0; tt < TT; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sh_[tt][i] = sl_[tt][i] = 0.0f;
    // scores += codes of k-step k (rows tt*16 + gq, + 8) x (high, remainder) of q*scale*f
    auto qk = [&](int k, const uint32_t (&bh)[2][2], const uint32_t (&bl)[2][2]) {
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        const uint32_t ka = (bkc ^ (16 * k)) + tt * 16 * ROWB;
        const uint32_t c0 = lds_u32(ka);
        const uint32_t c1 = lds_u32((ka ^ 64) + 8 * ROWB);
        const uint32_t d0 = c0 >> 8, d1 = c1 >> 8;
        uint32_t a[4] = {c0 & 0x000F000Fu, c1 & 0x000F000Fu, c0 & 0x00F000F0u, c1 & 0x00F000F0u};
        mma_f16_16816(sh_[tt], a, bh[0][0], bh[0][1]);
        mma_f16_16816(sl_[tt], a, bl[0][0], bl[0][1]);
        a[0] = d0 & 0x000F000Fu;
        a[1] = d1 & 0x000F000Fu;
        a[2] = d0 & 0x00F000F0u;
        a[3] = d1 & 0x00F000F0u;
        mma_f16_16816(sh_[tt], a, bh[1][0], bh[1][1]);
        mma_f16_16816(sl_[tt], a, bl[1][0], bl[1][1]);
      }
    };
    float bias_e = 0.0f, bias_o = 0.0f;  // sum of q*scale*f*zp over even / odd j (odd: / 16)
#pragma unroll
    for (int k = 0; k < KH; ++k) {
      const uint32_t kz = ((bq ^ (32 * (k >> 1)) ^ 64) ^ hx) + hoff + PG::kOffKz + 128 * k;
      const int4 z0 = lds_i4(kz + 16 * (k & 1));
      const int4 z1 = lds_i4(kz + 16 * ((k & 1) ^ 1));
      const int zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
      float ws[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ws[j] = w[8 * k + j] * ((j & 1) ? f16th : f);
        if (j & 1)
          bias_o = fmaf(ws[j], (float)zz[j], bias_o);
        else
          bias_e = fmaf(ws[j], (float)zz[j], bias_e);
      }
      uint32_t bh[2][2], bl[2][2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b0 = 2 * h;
        bh[h][0] = pack_f16(ws[b0], ws[b0 + 4]);
        bh[h][1] = pack_f16(ws[b0 + 1], ws[b0 + 5]);
        const float2 e0 = unpack_f16(bh[h][0]), e1 = unpack_f16(bh[h][1]);
        bl[h][0] = pack_f16(ws[b0] - e0.x, ws[b0 + 4] - e0.y);
        bl[h][1] = pack_f16(ws[b0 + 1] - e1.x, ws[b0 + 5] - e1.y);
      }
      qk(k, bh, bl);
      if constexpr (kSplit) {  // k-step k + 2, prepared by the lane 16 apart
        uint32_t rh[2][2], rl[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            rh[h][e] = __shfl_xor_sync(0xffffffffu, bh[h][e], 16);
            rl[h][e] = __shfl_xor_sync(0xffffffffu, bl[h][e], 16);
          }
        qk(k + 2, rh, rl);
      }
    }
    float bias = fmaf(16.0f, bias_o, bias_e);
    if constexpr (kSplit) bias += __shfl_xor_sync(0xffffffffu, bias, 16);
    bias += __shfl_xor_sync(0xffffffffu, bias, 1);
    bias += __shfl_xor_sync(0xffffffffu, bias, 2);
    const float bias0 = __shfl_sync(0xffffffffu, bias, 8 * q);
    const float bias1 = __shfl_sync(0xffffffffu, bias, 8 * q + 4);
    const float mul0 = __shfl_sync(0xffffffffu, finv, 8 * q) * scale_log2;
    const float mul1 = __shfl_sync(0xffffffffu, finv, 8 * q + 4) * scale_log2;

    // ---- online softmax for heads 2q, 2q+1
    float s[TT][4];
    // this lane's columns 2q, 2q+1 see the tokens below lim_a, lim_b (several query
    // tokens per sequence: causal lags; else both are the page's count)
    const int lim_a = MQ ? min(valid, to_end - lag_a) : valid, lim_b = MQ ? min(valid, to_end - lag_b) : valid;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const bool v0 = tt * 16 + gq < lim_a, v1 = tt * 16 + gq + 8 < lim_a;
      const bool w0 = tt * 16 + gq < lim_b, w1 = tt * 16 + gq + 8 < lim_b;
      s[tt][0] = v0 ? fmaf(sh_[tt][0] + sl_[tt][0], 0x1p24f, -bias0) * mul0 : -INFINITY;
      s[tt][1] = w0 ? fmaf(sh_[tt][1] + sl_[tt][1], 0x1p24f, -bias1) * mul1 : -INFINITY;
      s[tt][2] = v1 ? fmaf(sh_[tt][2] + sl_[tt][2], 0x1p24f, -bias0) * mul0 : -INFINITY;
      s[tt][3] = w1 ? fmaf(sh_[tt][3] + sl_[tt][3], 0x1p24f, -bias1) * mul1 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[tt][0], s[tt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[tt][1], s[tt][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // a column that has seen no token yet (several query tokens per
    // sequence) keeps an empty state instead of forming inf - inf
    const float r0 = MQ && n0 == -INFINITY ? 0.0f : n0, r1 = MQ && n1 == -INFINITY ? 0.0f : n1;
    const float a0 = ex2_approx(m0 - r0), a1 = ex2_approx(m1 - r1);
    m0 = n0;
    m1 = n1;
    uint32_t ph[TT][2], pl[TT][2];
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int tt = 0; tt < TT; ++tt) {
      const float p0 = ex2_approx(s[tt][0] - r0), p1 = ex2_approx(s[tt][1] - r1);
      const float p2 = ex2_approx(s[tt][2] - r0), p3 = ex2_approx(s[tt][3] - r1);
      ps0 += p0 + p2;
      ps1 += p1 + p3;
      const uint32_t h01 = pack_f16(p0, p1), h23 = pack_f16(p2, p3);
      const float2 f01 = unpack_f16(h01), f23 = unpack_f16(h23);
      ph[tt][0] = movmatrix_trans(h01);
      ph[tt][1] = movmatrix_trans(h23);
      pl[tt][0] = movmatrix_trans(pack_f16(p0 - f01.x, p1 - f01.y));
      pl[tt][1] = movmatrix_trans(pack_f16(p2 - f23.x, p3 - f23.y));
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
    float sum0 = ps0, sum1 = ps1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, off);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, off);
    }
    // ---- raw[c][h] = sum_t code_tc p_th, then o = alpha o + scale (raw - zp sum_p)
    // Byte sd of a token's word holds channels 2sd (low nibble: mma row gq) and
    // 2sd + 1 (high: row gq + 8); one byte permute puts two tokens' bytes in the
    // two halves, and the masks make them f16 subnormals code * 2^-24 (even
    // channel) or code * 2^-20 (odd). The rows of o therefore accumulate in those
    // units (zp sum_p scaled to match) and are scaled back when deposited.
    const float sum0e = sum0 * 0x1p-24f, sum1e = sum1 * 0x1p-24f;
    const float sum0o = sum0 * 0x1p-20f, sum1o = sum1 * 0x1p-20f;
#pragma unroll
    for (int oc = 0; oc < 2; ++oc) {
      float raw[4][4];
#pragma unroll
      for (int sd = 0; sd < 4; ++sd)
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[sd][i] = 0.0f;
#pragma unroll
      for (int tt = 0; tt < TT; ++tt) {
        const uint32_t va = (bvc ^ (32 * oc)) + tt * 16 * ROWB;  // tokens tt*16 + 2q + {0, 1, 8, 9}
        const uint32_t W0 = lds_u32(va);
        const uint32_t W1 = lds_u32(va ^ 64);
        const uint32_t W2 = lds_u32((va ^ 64) + 8 * ROWB);
        const uint32_t W3 = lds_u32(va + 8 * ROWB);
#pragma unroll
        for (int sd = 0; sd < 4; ++sd) {
          const uint32_t sel = (uint32_t)(sd | (sd << 4) | ((4 + sd) << 8) | ((4 + sd) << 12));
          const uint32_t x01 = prmt(W0, W1, sel), x89 = prmt(W2, W3, sel);
          uint32_t A[4] = {x01 & 0x000F000Fu, x01 & 0x00F000F0u, x89 & 0x000F000Fu, x89 & 0x00F000F0u};
          mma_f16_16816(raw[sd], A, ph[tt][0], ph[tt][1]);
          mma_f16_16816(raw[sd], A, pl[tt][0], pl[tt][1]);
        }
      }
      const uint32_t vs = (bvm ^ (32 * oc)) + PG::kOffVs + 256 * oc;  // channels 64oc + 8gq .. + 7
      const uint32_t vz = (bvm ^ (32 * oc) ^ 64) + PG::kOffVz + 256 * oc;
      const float4 s0 = lds_f4(vs), s1 = lds_f4(vs ^ 16);
      const int4 z0 = lds_i4(vz), z1 = lds_i4(vz ^ 16);
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const float zf[8] = {(float)z0.x, (float)z0.y, (float)z0.z, (float)z0.w,
                           (float)z1.x, (float)z1.y, (float)z1.z, (float)z1.w};
#pragma unroll
      for (int sd = 0; sd < 4; ++sd) {
        float* ot = o[4 * oc + sd];
        const int ce = 2 * sd, co = 2 * sd + 1;  // channels of rows g and g+8
        ot[0] = fmaf(a0, ot[0], sc[ce] * fmaf(-zf[ce], sum0e, raw[sd][0]));
        ot[1] = fmaf(a1, ot[1], sc[ce] * fmaf(-zf[ce], sum1e, raw[sd][1]));
        ot[2] = fmaf(a0, ot[2], sc[co] * fmaf(-zf[co], sum0o, raw[sd][2]));
        ot[3] = fmaf(a1, ot[3], sc[co] * fmaf(-zf[co], sum1o, raw[sd][3]));
      }
    }
  }

  __device__ __forceinline__ void deposit(float* st_acc, float* st_ml) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, q = lane & 3;
    float s0 = l0, s1 = l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const int h0 = 2 * q;
    if (lane < 4) {
      if (h0 < G) {
        st_ml[h0 * 2] = m0;
        st_ml[h0 * 2 + 1] = s0;
      }
      if (h0 + 1 < G) {
        st_ml[(h0 + 1) * 2] = m1;
        st_ml[(h0 + 1) * 2 + 1] = s1;
      }
    }
#pragma unroll
    for (int oc = 0; oc < 2; ++oc) {
#pragma unroll
      for (int sd = 0; sd < 4; ++sd) {
        const int c = 64 * oc + 8 * gq + 2 * sd;
        const float* ot = o[4 * oc + sd];
        if (h0 < G) {  // even channels in units of 2^-24, odd ones of 2^-20
          st_acc[h0 * D + stash_col<3>(h0, c)] = ot[0] * 0x1p24f;
          st_acc[h0 * D + stash_col<3>(h0, c + 1)] = ot[2] * 0x1p20f;
        }
        if (h0 + 1 < G) {
          st_acc[(h0 + 1) * D + stash_col<3>(h0 + 1, c)] = ot[1] * 0x1p24f;
          st_acc[(h0 + 1) * D + stash_col<3>(h0 + 1, c + 1)] = ot[3] * 0x1p20f;
        }
      }
    }
  }
  int lag_a = 0, lag_b = 0;  // causal lags of this lane's columns 2q, 2q+1
  // several query tokens per sequence: column c lags lag0 - c / gh tokens
  __device__ __forceinline__ void set_lags(int lag0, int gh) {
    const int q = threadIdx.x & 3;
    lag_a = lag0 - (2 * q) / gh;
    lag_b = lag0 - (2 * q + 1) / gh;
  }
  static constexpr int kStashSwz = 3;
};

// ------------------------------------------------------------------ the decode kernel
// One warp merges the W consumer warps' states of a unit from the stash
// (M = max_w m_w, f_w = 2^(m_w - M), o = sum_w f_w acc_w / sum_w f_w l_w) and
// writes heads 0..g-1 to o_dst ([g][D]) and, for a partial, their log-sum-exps
// (base 2) to lse_dst. Lane j owns channels j*D/32 .. (j+1)*D/32 - 1. All G
// heads are computed without branches (rows of heads >= g hold stale values
// and are not stored), so the loads and exponentials of every head overlap.
// Not inlined: the decode loop keeps its registers.
// With ROWS (column groups of several query tokens) head h is written to
// row (h / gh) * run + h % gh of o_dst instead of row h.
template <int D, int G, int W, int SWZ, bool ROWS = false>
__device__ __noinline__ void merge_stash_warp(const float* __restrict__ st_acc,
                                              const float* __restrict__ st_ml, int g,
                                              float* __restrict__ o_dst, float* __restrict__ lse_dst,
                                              int gh = 1, int run = 0, int hbeg = 0, int hstep = 1) {
  constexpr int CPL = D / 32;
  static_assert(CPL == 2 || CPL == 4, "head_dim 64 or 128");
  static_assert(SWZ < 2 || CPL == 4, "swizzles of bits 0-2 need four channels per lane");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (hstep > 1 && h % hstep != hbeg) continue;  // heads hbeg, hbeg + hstep, ... only
    float mw[W];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      mw[w] = st_ml[(w * G + h) * 2];
      M = fmaxf(M, mw[w]);
    }
    float Lsum = 0.0f, A[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) A[c] = 0.0f;
    // the word holding this lane's channels; SWZ 2 and 3 permute the four
    // channels inside it by (h >> 1) & 3
    const int col = stash_col<SWZ>(h, lane * CPL) & ~(CPL - 1);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = mw[w] == -INFINITY ? 0.0f : exp2f(mw[w] - M);
      Lsum = fmaf(st_ml[(w * G + h) * 2 + 1], f, Lsum);
      const float* src = st_acc + (w * G + h) * D + col;
      if constexpr (CPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) A[c] = fmaf(x[SWZ >= 2 ? (c ^ ((h >> 1) & 3)) : c], f, A[c]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        A[0] = fmaf(v.x, f, A[0]);
        A[1] = fmaf(v.y, f, A[1]);
      }
    }
    if (h < g) {
      const float inv = Lsum > 0.0f ? __frcp_rn(Lsum) : 0.0f;
      float* dst;
      if constexpr (ROWS)
        dst = o_dst + ((long long)(h / gh) * run + h % gh) * D + lane * CPL;
      else
        dst = o_dst + h * D + lane * CPL;
      if constexpr (CPL == 4)
        *reinterpret_cast<float4*>(dst) = make_float4(A[0] * inv, A[1] * inv, A[2] * inv, A[3] * inv);
      else
        *reinterpret_cast<float2*>(dst) = make_float2(A[0] * inv, A[1] * inv);
      if (lse_dst != nullptr && lane == 0) lse_dst[h] = Lsum > 0.0f ? M + log2f(Lsum) : -INFINITY;
    }
  }
}

// AP: the fused decode step's instantiation (each unit's new token stored by
// the block that reads the unit's last page, before that page is read); the
// plain decode's kernels are compiled without that code.
template <int KV, int D, int BS, int G, int NS, bool TC, bool MQ, bool AP = false>
__global__ void __launch_bounds__((consumer_warps<KV, TC, BS>() + 2) * 32, 1)
    paged_gqa_decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int kConsumerWarps = consumer_warps<KV, TC, BS>();
  constexpr int kThreads = (kConsumerWarps + 2) * 32;  // producer, consumers, merger
  using SM = Smem<KV, D, BS, G, NS, kConsumerWarps, TC>;
  using PG = PageGeom<KV, D, BS>;
  using Cons = typename std::conditional<
      TC,
      typename std::conditional<
          KV == PA_KV_BF16, MmaConsumerBf16<D, BS, G>,
          typename std::conditional<
              KV == PA_KV_UINT8, MmaConsumerU8<BS, G>,
              typename std::conditional<KV == PA_KV_FP8, MmaConsumerFp8<BS, G>, MmaConsumerU4<BS, G>>::type>::type>::type,
      FmaConsumer<KV, D, BS, G>>::type;
  static_assert(!TC || KV == PA_KV_BF16 || D == 128,
                "tensor-core consumers: bf16 pages, or quantised pages of head_dim 128");
  constexpr int NST = SM::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled TMA destinations
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kOffBars);
  uint64_t* empty = full + NST;
  uint64_t* qfull = empty + NST;
  uint64_t* qempty = qfull + 2;
  uint64_t* deposited = qempty + 2;  // every consumer warp has stashed the unit
  uint64_t* merged = deposited + 1;   // the merger has read the stash (free again)
  uint64_t* appended = merged + 1;    // fused step: this window's new tokens are stored
  int32_t* stage_flag = reinterpret_cast<int32_t*>(smem + SM::kOffFlags);
  Seg* segs = reinterpret_cast<Seg*>(smem + SM::kOffSegs);
  long long* plan = reinterpret_cast<long long*>(smem + SM::kOffPlan);
  int32_t* phys_s = reinterpret_cast<int32_t*>(smem + SM::kOffPhys);
  uint8_t* qslots = smem + SM::kOffQ;
  float* stash_acc = reinterpret_cast<float*>(smem + SM::kOffStash);
  float* stash_ml = reinterpret_cast<float*>(smem + SM::kOffStashML);
  float* pbuf_all = reinterpret_cast<float*>(smem + SM::kOffPbuf);
  uint8_t* stages = smem + SM::kOffStages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.pool.num_kv_heads;
  const int g = p.group;
  const long long Gc = gridDim.x, cta = blockIdx.x;
  __shared__ int warp_tot[32];
  __shared__ volatile int abort_flag;
  __shared__ int issued_n[NST];  // last fill issued per stage (drain on abort)
  __shared__ int q_issued[2];    // last q segment index issued per slot

  // Launched with programmatic stream serialization: let the combine kernel
  // be scheduled early; write no global memory and read no page before the
  // preceding kernel in the stream has completed. With early_plan the caller
  // vouches that the preceding kernel writes neither the lengths nor the
  // block table, so the read-only planning below (lengths, slice, segment
  // list, block-table entries) overlaps it.
  pdl_launch_dependents();
  // the TMA descriptor is fetched while the plan runs
  if (tid == 0 && p.maps.valid) prefetch_tensormap(&p.maps.rec);
  bool waited = false;
  if (!p.early_plan) {
    pdl_wait();
    waited = true;
  }

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      issued_n[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kConsumerWarps);
    }
    mbar_init(deposited, kConsumerWarps);
    mbar_init(merged, 1);
    if constexpr (AP) mbar_init(appended, kConsumerWarps);
    abort_flag = 0;
    q_issued[0] = q_issued[1] = -1;
    fence_mbar_init();
  }

  // ---- plan: the cost line, this slice, and where it starts. Checked
  // lengths of the first kLensSmem sequences are kept in shared memory (in
  // the merge stash, idle until the consumer warps start) for a second pass
  // and the first window's segment list.
  int* lens_sm = reinterpret_cast<int*>(stash_acc);
  constexpr int kLensSmem = (int)(SM::kStashAccBytes / 4);
  // With at most one sequence per thread (the usual case) one block scan
  // gives every sequence's first page, so the slice start and the prefix
  // CTA 0 publishes need no second pass over the lengths.
  const bool one_pass = p.batch <= kThreads;
  if (tid == 0) plan[0] = -1;
  int my_pages = 0, my_incl = 0;
  long long npages_all = 0;
  if (p.batch <= 32) {
    // at most 32 sequences: every warp loads and scans the lengths itself
    // (the loads hit L1 after the first), so no block barrier is needed;
    // warp 0's lanes hold the per-sequence values the one-pass plan uses
    const int len = lane < p.batch ? vlen_checked<MQ>(p, lane, cta == 0 && warp == 0) : 0;
    if (warp == 0 && lane < p.batch) lens_sm[lane] = len;
    const int span = unit_span((len + BS - 1) / BS, p.unit_cost);
    int x = span;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    my_incl = warp == 0 ? x : 0;
    my_pages = warp == 0 ? span : 0;
    npages_all = __shfl_sync(0xffffffffu, x, 31);
  } else {
    int part = 0;
    for (int b = tid; b < p.batch; b += kThreads) {
      const int len = vlen_checked<MQ>(p, b, cta == 0);
      if (b < kLensSmem) lens_sm[b] = len;
      part += unit_span((len + BS - 1) / BS, p.unit_cost);
    }
    int tot;
    my_incl = block_incl_scan(part, warp_tot, tot);
    my_pages = part;
    npages_all = tot;
  }
  // T: length of the cost line; this thread block's slice is [s_i, e_i)
  const long long T = npages_all * Hkv;
  const bool small = line_small(T, Gc);
  const long long s_i = slice_start(cta, T, Gc, small), e_i = slice_start(cta + 1, T, Gc, small);
  // Ring stages in use (of the NST allocated): about one per 8 pages of a
  // slice, 16 to 24. Short slices run better with fewer pages in flight (the
  // first copies land sooner and HBM queues stay short); long ones need the
  // depth. The same for every thread block of the launch. A multiple of the
  // consumer warp count, so that pages k and k + nst, which share a stage,
  // belong to the same consumer warp: a warp then starts waiting for a fill
  // only after it has itself released the fill before, and its parity wait
  // can never mistake an older phase still in flight for the one it wants.
  // Rounded up (NST is a multiple of kConsumerWarps, so the result stays
  // within the ring and is at least one warp count).
  const int nst = (int)min((long long)NST, (max((long long)min(NST, kConsumerWarps), min((long long)NST, max(16LL, min(24LL, (small ? (long long)((unsigned)T / (unsigned)Gc) : T / Gc) / 8)))) +
                                            kConsumerWarps - 1) /
                                               kConsumerWarps * kConsumerWarps);
  // every thread block finds the sequence holding its first page
  if (one_pass) {
    const long long lo = (long long)(my_incl - my_pages) * Hkv, hi = (long long)my_incl * Hkv;
    if (tid < p.batch && s_i >= lo && s_i < hi) {
      plan[0] = tid;
      plan[1] = lo;
    }
  } else {
    int running = 0;
    for (int base = 0; base < p.batch; base += kThreads) {
      const int b = base + tid;
      const int n = b < p.batch ? unit_span(((b < kLensSmem ? lens_sm[b] : vlen_checked<MQ>(p, b, false)) + BS - 1) / BS, p.unit_cost) : 0;
      int tot;
      const int incl = block_incl_scan(n, warp_tot, tot);
      const long long lo = (long long)(running + incl - n) * Hkv;
      const long long hi = (long long)(running + incl) * Hkv;
      if (b < p.batch && s_i >= lo && s_i < hi) {
        plan[0] = b;
        plan[1] = lo;
      }
      running += tot;
      if (cta != 0) {
        __syncthreads();
        const bool found = plan[0] >= 0;
        __syncthreads();
        if (found) break;
      }
    }
  }
  // CTA 0 publishes the per-sequence cost prefix for the combine kernel (and,
  // with the in-kernel merge, zero rows for empty sequences): global writes,
  // so after the wait. lens_sm is still intact (the consumers have not
  // started).
  bool published = false;
  auto wait_and_publish = [&]() {
    if (published) return;
    published = true;
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    if (cta != 0) return;
    if (one_pass) {
      if (tid < p.batch) p.pre_cost[tid] = my_incl - my_pages;
      if (tid == p.batch - 1) p.pre_cost[p.batch] = my_incl;
    } else {
      int running = 0;
      for (int base = 0; base < p.batch; base += kThreads) {
        const int b = base + tid;
        const int n = b < p.batch ? unit_span(((b < kLensSmem ? lens_sm[b] : vlen_checked<MQ>(p, b, false)) + BS - 1) / BS, p.unit_cost) : 0;
        int tot;
        const int incl = block_incl_scan(n, warp_tot, tot);
        if (b < p.batch) p.pre_cost[b] = running + incl - n;
        if (b == p.batch - 1) p.pre_cost[p.batch] = running + incl;
        running += tot;
      }
    }
    if (p.batch == 0 && tid == 0) p.pre_cost[0] = 0;
    if (!MQ && p.fused) {
      // rows of empty sequences: no slice holds a page of them
      const int row_elems = p.num_q_heads * D;
      for (int b = 0; b < p.batch; ++b) {
        const int len = b < kLensSmem ? lens_sm[b] : vlen_checked<MQ>(p, b, false);
        if (len == 0)
          for (int e = tid; e < row_elems; e += kThreads) p.out[(long long)b * row_elems + e] = 0.0f;
      }
    }
    __syncthreads();
  };
  if (!p.early_plan) wait_and_publish();
  __syncthreads();
  if (s_i >= e_i) {  // no pages for this thread block
    wait_and_publish();
    return;
  }

  long long cur_b = plan[0], cur_base = plan[1];  // sequence holding `pos` and its start on the line
  long long pos = s_i;       // cost-line position of the window
  int k_done = 0;            // real pages of the slice in earlier windows
  int seg_counter = 0;      // segments started so far (q slot ring index)
  bool lens_cached = true;  // lens_sm valid until the consumer warps write the stash
  uint64_t pol = policy_evict_first();
  Cons cons;  // consumer warps' online-softmax state; persists across windows
  int n_dep = 0;  // units this warp has deposited (phase of `merged` to wait for)
  int win = 0;    // windows done (phase of `appended` to wait for)
  constexpr bool fuse_append = AP && !MQ;  // the fused decode step's kernels only

  while (pos < e_i) {
    // ---- build this window's segment list (warp 0)
    if (warp == 0) {
      int nseg = 0;
      int kcount = k_done;  // real pages of the slice before the next segment
      long long b0 = cur_b, base0 = cur_base, wpos = pos;
      const long long wlim = min(e_i, pos + (long long)kMaxWinPages);
      bool done = false;
      while (!done && b0 < p.batch) {
        const long long bb = b0 + lane;
        const int len = bb >= p.batch ? 0
                        : (lens_cached && bb < kLensSmem) ? lens_sm[bb]
                                                          : vlen_checked<MQ>(p, (int)bb, false);
        const int n = (len + BS - 1) / BS;  // real pages per unit
        const int cn = unit_span(n, p.unit_cost);  // its span on the cost line
        int x = cn;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const long long my_base = base0 + (long long)(x - cn) * Hkv;
        const long long my_end = my_base + (long long)cn * Hkv;
        const bool overl = cn > 0 && my_end > wpos && my_base < wlim && bb < p.batch;
        unsigned mask = __ballot_sync(0xffffffffu, overl);
        while (mask) {
          const int src = __ffs(mask) - 1;
          mask &= mask - 1;
          const long long sb = b0 + src;
          const long long sbase = __shfl_sync(0xffffffffu, my_base, src);
          const int sn = __shfl_sync(0xffffffffu, n, src);
          const int scn = __shfl_sync(0xffffffffu, cn, src);
          const int slen = __shfl_sync(0xffffffffu, len, src);
          // (both offsets below T; sbase < wlim)
          const long long off_lo = wpos > sbase ? wpos - sbase : 0, off_hi = wlim - 1 - sbase;
          const int h_lo = (int)(small ? (long long)((unsigned)off_lo / (unsigned)scn) : off_lo / scn);
          const int h_hi = (int)min((long long)Hkv - 1,
                                    small ? (long long)((unsigned)off_hi / (unsigned)scn) : off_hi / scn);
          for (int h = h_lo; h <= h_hi && !done; ++h) {
            // unit h: real pages [us, ure), then phantom positions up to ue
            const long long us = sbase + (long long)h * scn, ure = us + sn, ue = us + scn;
            const long long lo = max(us, wpos), hic = min(ue, wlim);
            if (lo >= hic) continue;
            const long long hi = min(ure, wlim);
            if (lo < hi) {
              if (lane == 0) {
                Seg sg;
                sg.b = (int)sb;
                sg.h = h;
                sg.lp0 = (int)(lo - us);
                sg.npages = (int)(hi - lo);
                sg.k0 = kcount;
                sg.len = slen;
                sg.us = us;
                const long long first = owner_of(us, T, Gc, small), last = owner_of(ure - 1, T, Gc, small);
                sg.slot = first == last ? -1 : (int)(cta + sb * Hkv + h);
                // a unit's pages are contiguous within a slice: a run that starts
                // after both the unit's and the slice's first page continues the
                // previous window; one that stops before both ends goes on
                sg.flags = (lo > us && lo > s_i ? kContPrev : 0) | (hi < ure && hi < e_i ? kContNext : 0);
                segs[nseg] = sg;
              }
              ++nseg;
              kcount += (int)(hi - lo);
            }
            wpos = hic;
            if (hic >= wlim || nseg == kMaxSegs) {
              done = true;
              // the next window resumes at the sequence holding wpos
              if (wpos >= sbase + (long long)scn * Hkv) {
                cur_b = sb + 1;
                cur_base = sbase + (long long)scn * Hkv;
              } else {
                cur_b = sb;
                cur_base = sbase;
              }
            }
          }
        }
        if (!done) {
          const int tot = __shfl_sync(0xffffffffu, x, 31);
          base0 += (long long)tot * Hkv;
          b0 += 32;
        }
      }
      if (lane == 0) {
        plan[2] = nseg;
        plan[3] = wpos;
        plan[4] = cur_b;
        plan[5] = cur_base;
        plan[6] = kcount;
      }
    }
    __syncthreads();
    const int nseg = (int)plan[2];
    const long long wend = plan[3];
    cur_b = plan[4];
    cur_base = plan[5];
    // the window's real pages are kw0 .. kw1 - 1 of the slice
    const int kw0 = k_done, kw1 = (int)plan[6];

    {
      // the window's page records -> shared memory: the block-table entry
      // of each page, checked and turned into its record index (block * Hkv
      // + head; -1 for an entry outside the pool), by every thread with
      // kStageLoads independent loads in flight (one round trip for windows
      // of up to kStageLoads * kThreads pages)
      constexpr int kStageLoads = 4;
      const int nwin = kw1 - kw0;
      // the window's q rows -> L2 too (a hint, safe before the wait), so
      // that the producer's copies of them land fast
      if (warp == 0) {
        for (int qi = lane; qi < nseg; qi += 32) {
          if constexpr (MQ) {
            for (int c = 0; c < unit_cols<MQ>(p, segs[qi].b); c += p.g_heads)
              prefetch_l2_bulk(p.q + unit_row<MQ>(p, segs[qi].b, segs[qi].h, c) * D, p.g_heads * D * 2);
          } else {
            const uint16_t* qsrc = p.q + ((long long)segs[qi].b * p.num_q_heads + (long long)segs[qi].h * g) * D;
            prefetch_l2_bulk(qsrc, g * D * 2);
          }
        }
      }
      for (int i0 = 0; i0 < nwin; i0 += kStageLoads * kThreads) {
        int v[kStageLoads];
#pragma unroll
        for (int u = 0; u < kStageLoads; ++u) {
          const int i = i0 + u * kThreads + tid;
          v[u] = 0;
          if (i < nwin) {
            const int k = kw0 + i;
            int lo = 0, hi = nseg - 1;  // last segment starting at or before k
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (segs[mid].k0 <= k) lo = mid; else hi = mid - 1;
            }
            const Seg& sg = segs[lo];
            const int phys = p.block_table[(long long)seq_of<MQ>(p, sg.b) * p.max_blocks + sg.lp0 + (k - sg.k0)];
            v[u] = (phys < 0 || phys >= p.pool.num_blocks) ? -1 : phys * Hkv + sg.h;
          }
        }
#pragma unroll
        for (int u = 0; u < kStageLoads; ++u) {
          const int i = i0 + u * kThreads + tid;
          if (i < nwin) phys_s[i] = v[u];
        }
      }
    }
    __syncthreads();
    wait_and_publish();  // first window only: pages and outputs follow

    // merge the stash of unit sg into its row or partial: heads hbeg,
    // hbeg + hstep, ... (all of them with the defaults)
    auto merge_unit = [&](const Seg& sg, int hbeg, int hstep) {
      const long long row0 = (long long)sg.b * p.num_q_heads + (long long)sg.h * g;
      if constexpr (MQ) {
        // rows of the column group: g_heads per query token, a token's rows
        // num_q_heads apart
        const int cols = unit_cols<MQ>(p, sg.b);
        if (sg.slot < 0)
          merge_stash_warp<D, G, kConsumerWarps, Cons::kStashSwz, true>(
              stash_acc, stash_ml, cols, p.out + unit_row<MQ>(p, sg.b, sg.h, 0) * D, nullptr, p.g_heads,
              p.num_q_heads, hbeg, hstep);
        else
          merge_stash_warp<D, G, kConsumerWarps, Cons::kStashSwz>(
              stash_acc, stash_ml, cols, p.part_o + (long long)sg.slot * g * D, p.part_lse + (long long)sg.slot * g,
              1, 0, hbeg, hstep);
      } else if (sg.slot < 0) {
        merge_stash_warp<D, G, kConsumerWarps, Cons::kStashSwz>(stash_acc, stash_ml, g, p.out + row0 * D, nullptr,
                                                                1, 0, hbeg, hstep);
      } else {
        merge_stash_warp<D, G, kConsumerWarps, Cons::kStashSwz>(stash_acc, stash_ml, g,
                                                                p.part_o + (long long)sg.slot * g * D,
                                                                p.part_lse + (long long)sg.slot * g, 1, 0, hbeg, hstep);
      }
    };
    // The slice's last unit: its merge ends this thread block's critical
    // path, and the consumer warps have no pages left, so they share it with
    // the merger warp (heads split over the kConsumerWarps + 1 warps), then
    // meet at named barrier 1.
    constexpr int kMergeWarps = kConsumerWarps + 1;
    const int last_si = wend >= e_i ? nseg - 1 : -1;

    if (warp == 0) {
      // ---------------------------------------------------------- producer
      // (2) issue in sub-batches, lane j taking page k + j. A sub-batch holds
      // at most one page per stage (<= nst pages): the previous fill of each
      // lane's stage was issued by an earlier sub-batch, after the release of
      // the fill before it, so each parity wait below sees its barrier at most
      // one phase behind. (Two lanes on one stage could see a barrier two
      // phases behind, take its parity for "released" and overwrite a stage
      // still in use.) A sub-batch never crosses the start of a segment: the
      // segment's q goes out first (lane 0).
      // q of segment qi into its slot (lane 0). The slot is free once every
      // consumer warp has begun segment qi - 2; without `block` the copy is
      // only sent if it already is.
      auto send_q = [&](int qi, bool block) -> bool {
        const int gs = seg_counter + qi;
        const int slot = gs & 1;
        if (gs >= 2 && !abort_flag) {
          const uint32_t par = ((gs >> 1) - 1) & 1;
          if (!block) {
            if (!mbar_try_wait(&qempty[slot], par)) return false;
          } else if (!mbar_wait_bounded(&qempty[slot], par)) {
            set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
        }
        const Seg& qs = segs[qi];
        if (abort_flag) {
          mbar_arrive(&qfull[slot]);
        } else if constexpr (MQ) {
          // one run of g_heads rows per query token of the column group
          const int cols = unit_cols<MQ>(p, qs.b);
          q_issued[slot] = gs;
          mbar_arrive_expect_tx(&qfull[slot], cols * D * 2);
          for (int c = 0; c < cols; c += p.g_heads)
            bulk_g2s(qslots + slot * SM::kQBytes + c * D * 2, p.q + unit_row<MQ>(p, qs.b, qs.h, c) * D,
                     p.g_heads * D * 2, &qfull[slot], pol);
        } else {
          const uint16_t* qsrc = p.q + ((long long)qs.b * p.num_q_heads + (long long)qs.h * g) * D;
          q_issued[slot] = gs;
          mbar_arrive_expect_tx(&qfull[slot], g * D * 2);
          bulk_g2s(qslots + slot * SM::kQBytes, qsrc, g * D * 2, &qfull[slot], pol);
        }
        return true;
      };
      int qseg = 0;    // segments whose first page the issue has reached
      int q_sent = 0;  // segments whose q has been sent (lane 0's count)
      bool tails_released = false;  // fused step: the consumers' stores of this window are done
      for (int k = kw0; k < kw1;) {
        if (qseg < nseg && segs[qseg].k0 == k) {
          if (lane == 0 && q_sent == qseg) {
            send_q(qseg, true);
            ++q_sent;
          }
          ++qseg;
          __syncwarp();
        }
        // the next segment's q goes out as soon as its slot is free, a ring's
        // worth of pages before the consumers need it
        if (lane == 0 && q_sent == qseg && q_sent < nseg && send_q(q_sent, false)) ++q_sent;
        int kend = min(kw1, k + (nst < 32 ? nst : 32));
        if (qseg < nseg) kend = min(kend, segs[qseg].k0);
        if (fuse_append && !tails_released) {
          // this sub-batch lies in segment qseg - 1: if it holds that unit's
          // last page, the consumers must have stored the new token first
          const Seg& cs = segs[qseg - 1];
          if (cs.len > 0 && cs.lp0 + cs.npages == (cs.len + BS - 1) / BS && kend == cs.k0 + cs.npages) {
            if (!abort_flag && !mbar_wait_bounded(appended, win & 1)) {
              set_error(p.pool.err, PA_DEVERR_TIMEOUT);
              abort_flag = 1;
            }
            tails_released = true;
          }
        }
        const int kk = k + lane;
        if (kk < kend) {
          const int rec = phys_s[kk - kw0];  // record index, -1 for a bad table entry
          const int stage = kk % nst;
          const int n = kk / nst;
          bool ok = true;
          if (n >= 1 && !abort_flag) ok = mbar_wait_bounded(&empty[stage], (n - 1) & 1);
          if (!ok) {
            set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
          if (rec < 0 || abort_flag) {
            if (!abort_flag) set_error(p.pool.err, PA_DEVERR_BLOCK_TABLE);
            stage_flag[stage] = 1;
            mbar_arrive(&full[stage]);
          } else {
            stage_flag[stage] = 0;
            uint8_t* dst = stages + (size_t)stage * PG::kStageBytes;
            const long long page = rec;
            issued_n[stage] = n;
            mbar_arrive_expect_tx(&full[stage], PG::kStageBytes);
            if (TC && KV != PA_KV_BF16) {
              // the whole record as one box of 128-byte rows, swizzled
              tma_load_2d(dst, &p.maps.rec, 0, (int)(page * p.maps.rows_per_page), &full[stage], pol);
            } else if (TC) {
              // one box of 64 channels x (K and V rows) per half, swizzled
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf)
                tma_load_2d(dst + hf * 2 * BS * 128, &p.maps.rec, hf * 64, (int)(page * 2 * BS),
                            &full[stage], pol);
            } else {
              // the whole record, unswizzled
              bulk_g2s(dst, page_of(p.pool.k, page, p.pool.stride), PG::kStageBytes, &full[stage], pol);
            }
          }
        }
        __syncwarp();
        k = kend;
      }
    } else if (warp <= kConsumerWarps) {
      // ---------------------------------------------------------- consumers
      const int cw = warp - 1;
      float* pbuf = pbuf_all + cw * BS * G;
      if constexpr (fuse_append) {
        // fused decode step: store the new token of every unit whose last page
        // lies in this window (this block owns that page), then release the
        // window's last pages to the producer. The stores go out through the
        // generic proxy and the pages come in by TMA: fence the two.
        for (int si = 0; si < nseg; ++si) {
          const Seg& sg = segs[si];
          if (sg.len <= 0 || sg.lp0 + sg.npages != (sg.len + BS - 1) / BS) continue;  // not the unit's last page
          const int rec = phys_s[sg.k0 + sg.npages - 1 - kw0];
          if (rec >= 0)
            append_unit_tail<KV, BS>(p.pool, rec, seq_of<MQ>(p, sg.b), sg.h, sg.len, p.k_new, p.v_new,
                                     cw * 32 + lane, kConsumerWarps * 32);
        }
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) mbar_arrive(appended);
      }
      if (pos == s_i) {
        // warm the instruction cache while the first pages are in flight: the
        // deposit runs once per unit, and its first run would otherwise fetch
        // instructions mid-stream, with memory saturated. A dry run into this
        // warp's own stash rows (free: the planning is done with them).
        Cons dry;
        dry.begin_unit(reinterpret_cast<const uint16_t*>(qslots), g, p.scale_log2);
        dry.deposit(stash_acc + cw * G * D, stash_ml + cw * G * 2);
      }
      for (int si = 0; si < nseg; ++si) {
        const Seg sg = segs[si];
        const int gs = seg_counter + si;
        const int slot = gs & 1;
        bool ok = abort_flag == 0 && mbar_wait_bounded(&qfull[slot], (gs >> 1) & 1);
        if (!ok && abort_flag == 0) {
          if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        if (!(sg.flags & kContPrev)) {
          cons.begin_unit(reinterpret_cast<const uint16_t*>(qslots + slot * SM::kQBytes), unit_cols<MQ>(p, sg.b),
                          p.scale_log2);
          if constexpr (MQ) cons.set_lags(unit_lag0<MQ>(p, sg.b), p.g_heads);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[slot]);
        // my pages: k = k0 + i with k % W == cw
        const int kfirst = sg.k0 + ((cw - sg.k0 % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
        // ring position of k, advanced without dividing (kConsumerWarps <= nst)
        int stage = kfirst % nst, n = kfirst / nst;
        for (int k = kfirst; k < sg.k0 + sg.npages; k += kConsumerWarps) {
          bool okp = abort_flag == 0 && mbar_wait_bounded(&full[stage], n & 1);
          if (!okp && abort_flag == 0) {
            if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
          if (okp && stage_flag[stage] == 0) {
            const int lp = sg.lp0 + (k - sg.k0);
            const int valid = min(BS, sg.len - lp * BS);
            cons.template page<MQ>(stages + (size_t)stage * PG::kStageBytes, valid, pbuf, sg.len - lp * BS);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
          stage += kConsumerWarps;
          if (stage >= nst) {
            stage -= nst;
            ++n;
          }
        }
        if (sg.flags & kContNext) continue;  // the run goes on in the next window
        // ---- hand this warp's state of the unit to the merger warp and go on
        // with the next unit's pages (waiting for the other warps here would
        // idle every warp until the unit's slowest page had landed and been
        // merged, and the ring would run dry)
        if (n_dep > 0) {
          // the stash is free once the previous unit's merge has read it
          const bool okm = mbar_wait_bounded(merged, (n_dep - 1) & 1);
          if (!okm && abort_flag == 0) {
            if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
        }
        ++n_dep;
        cons.deposit(stash_acc + cw * G * D, stash_ml + cw * G * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(deposited);  // release: the stash rows above
        if (si == last_si) {
          const bool okd = mbar_wait_bounded(deposited, (n_dep - 1) & 1);  // every warp's state is in
          if (!okd && abort_flag == 0) {
            if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
          merge_unit(sg, cw, kMergeWarps);
          if (p.fused) __threadfence();  // this warp's partial rows before the merger's ticket
          named_bar_sync(1, kMergeWarps * 32);
        }
      }
    } else {
      // ---------------------------------------------------------- merger
      // One warp merges each finished unit from the stash (in segment order,
      // as the consumers deposit them) and writes its row or partial.
      if (pos == s_i) {
        // instruction-cache warm-up while the first pages are in flight: a
        // dry merge that stores nothing (no heads); what it reads is discarded
        merge_stash_warp<D, G, kConsumerWarps, Cons::kStashSwz>(stash_acc, stash_ml, 0, p.out, nullptr);
      }
      for (int si = 0; si < nseg; ++si) {
        const Seg sg = segs[si];
        if (sg.flags & kContNext) continue;
        const bool okd = mbar_wait_bounded(deposited, n_dep & 1);
        if (!okd && abort_flag == 0) {
          if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        ++n_dep;
        const long long row0 = (long long)sg.b * p.num_q_heads + (long long)sg.h * g;
        if (si == last_si) {
          merge_unit(sg, kConsumerWarps, kMergeWarps);
          named_bar_sync(1, kMergeWarps * 32);
        } else {
          merge_unit(sg, 0, 1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merged);  // the stash may be overwritten
        if (!MQ && sg.slot >= 0 && p.fused) {
          // the last slice to finish this unit merges its partials (threadfence
          // reduction: partials are fenced before the ticket is taken)
          __threadfence();
          __syncwarp();
          UnitSlices usl;
          usl.n = (sg.len + BS - 1) / BS;
          usl.us = sg.us;
          usl.T = T;
          usl.G = Gc;
          usl.small = small;
          usl.first = owner_of(usl.us, T, Gc, small);
          usl.last = owner_of(usl.us + usl.n - 1, T, Gc, small);
          const long long u = (long long)sg.b * Hkv + sg.h;
          int last_slice = 0;
          if (lane == 0) {
            const unsigned long long tag = p.epoch << 24;
            const unsigned long long cnt = (unsigned long long)usl.count();  // >= 2: the unit is split
            unsigned long long* t = p.tickets + u;
            // first guess: every other slice is done (this call's tag, cnt - 1),
            // so the last slice, the one on the critical path, takes its ticket
            // in one round trip; a wrong guess returns the value to retry with
            unsigned long long old = tag | (cnt - 1), assumed;
            unsigned long long mine;
            do {
              assumed = old;
              const unsigned long long done = (assumed >> 24) == p.epoch ? (assumed & 0xFFFFFFull) : 0ull;
              mine = done + 1;
              old = atomicCAS(t, assumed, tag | mine);
            } while (old != assumed);
            last_slice = mine == cnt ? 1 : 0;
          }
          last_slice = __shfl_sync(0xffffffffu, last_slice, 0);
          if (last_slice) {
            __threadfence();
            merge_unit_partials<D>(usl, u, row0, g, p.part_o, p.part_lse, p.out, lane, 32);
            // every slice of the unit has taken its ticket: clear it, so that a
            // replay of this very launch (a CUDA graph keeps its epoch) starts
            // from zero again
            if (lane == 0) *reinterpret_cast<volatile unsigned long long*>(p.tickets + u) = 0ull;
          }
        }
      }
    }
    seg_counter += nseg;
    lens_cached = false;
    pos = wend;
    k_done = kw1;
    if constexpr (fuse_append) ++win;
    __syncthreads();
  }
  // every issued copy was waited on by a consumer (or the abort path skipped
  // it); drain any that a timed-out consumer left behind
  if (abort_flag && tid == 0) {
    for (int i = 0; i < NST; ++i)
      if (issued_n[i] >= 0) mbar_wait_bounded(&full[i], issued_n[i] & 1, 400000000LL);
    for (int i = 0; i < 2; ++i)
      if (q_issued[i] >= 0) mbar_wait_bounded(&qfull[i], (q_issued[i] >> 1) & 1, 400000000LL);
  }
}

// ------------------------------------------------------------------ split-KV combine
// One thread block per unit (b, j). Units whose pages all fell in one slice
// were written by the decode kernel; empty sequences get zero rows; the rest
// merge their partials: M = max_s lse_s, w_s = 2^(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s (the same algebra as the online-softmax
// update, applied to whole partial states).
//
// Everything that depends only on the lengths (the unit's page range, its
// slices and which of them hold a partial) is worked out before the wait on
// the decode kernel when the caller allows reading the lengths early (they
// are inputs the decode kernel never writes); after the wait one round of
// loads fetches every partial of the unit: a thread owns four channels of
// one head and issues its loads for all slices back to back.
// With MQ (several query tokens per sequence) the units are those of the
// virtual sequences (see DecodeParams): lengths come from sequence b / n_cg
// and column c of a unit goes to its own row.
// Launched with kCombineThreads threads, one four-channel quad of the unit's
// columns each (at most 8 columns of 128 channels). (A four-warp variant at
// 112 registers, which fits beside a decode thread block on one SM, measured
// 0.3 us faster back to back but 0.5 us slower per isolated call, and made
// the decode step no faster.)
constexpr int kCombineThreads = 256;
template <int D, bool MQ = false>
__global__ void __launch_bounds__(kCombineThreads)
    splitkv_combine_kernel(const int32_t* seq_lens, const int32_t* pre_cost, const float* part_o,
                           const float* part_lse, float* out, int batch, int num_kv_heads, int group,
                           int num_q_heads, int num_ctas, int block_size, int max_blocks, int unit_cost,
                           int lens_early, int n_q = 1, int n_cg = 1, int tpg = 1, int g_heads = 1) {
  constexpr int kMaxSl = 64;  // slices handled from the precomputed mask; more go round again
  __shared__ long long sh_sum[2][8];
  pdl_launch_dependents();
  const int u = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = u / num_kv_heads, j = u % num_kv_heads;
  // pre: the sequence's start on the cost line (per head); n: its pages; cn:
  // its span per head; T: the line's length (the decode kernel's partition)
  long long pre = 0, n = 0, cn = 0, T = 0;
  auto unit_range = [&](bool from_lens) {
    if (from_lens) {
      // spans of every sequence and of those before b, from the lengths
      // (invalid lengths count as empty, as in the decode kernel)
      long long all = 0, before = 0;
      for (int x = tid; x < batch; x += blockDim.x) {
        const int len = seq_lens[MQ ? x / n_cg : x];
        const int np =
            (len < 0 || (long long)len > (long long)max_blocks * block_size) ? 0 : (len + block_size - 1) / block_size;
        const int span = unit_span(np, unit_cost);
        all += span;
        if (x < b) before += span;
        if (x == b) n = np;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        all += __shfl_xor_sync(0xffffffffu, all, o);
        before += __shfl_xor_sync(0xffffffffu, before, o);
      }
      if (lane == 0) {
        sh_sum[0][warp] = all;
        sh_sum[1][warp] = before;
      }
      __syncthreads();
      all = before = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        all += sh_sum[0][w];
        before += sh_sum[1][w];
      }
      // n: the thread that saw b shares it
      __syncthreads();
      if (b % (int)blockDim.x == tid) sh_sum[0][0] = n;
      __syncthreads();
      n = sh_sum[0][0];
      cn = unit_span((int)n, unit_cost);
      pre = before;
      T = all * num_kv_heads;
    } else {
      pre = pre_cost[b];
      cn = pre_cost[b + 1] - pre;
      n = cn > 0 ? cn - unit_cost : 0;
      T = (long long)pre_cost[batch] * num_kv_heads;
    }
  };
  UnitSlices usl;
  unsigned long long mask0 = 0;  // first round's slices that hold a partial
  auto unit_slices = [&]() {
    usl.us = pre * num_kv_heads + (long long)j * cn;
    usl.n = n;
    usl.T = T;
    usl.G = num_ctas;
    usl.small = line_small(T, num_ctas);
    usl.first = n > 0 ? owner_of(usl.us, T, num_ctas, usl.small) : 0;
    usl.last = n > 0 ? owner_of(usl.us + n - 1, T, num_ctas, usl.small) : 0;
    const int cnt = (int)min((long long)kMaxSl, usl.last - usl.first + 1);
    for (int i = 0; i < cnt && usl.first != usl.last; ++i)
      if (usl.has_part(usl.first + i)) mask0 |= 1ull << i;
  };
  if (lens_early) {
    unit_range(true);
    unit_slices();
  }
  pdl_wait();
  if (!lens_early) {
    unit_range(false);
    unit_slices();
  }
  const long long row0 = (long long)b * num_q_heads + (long long)j * group;
  // the unit's columns and the output row of column c
  const int cols = MQ ? min(tpg, n_q - (b % n_cg) * tpg) * g_heads : group;
  auto out_row = [&](int c) -> long long {
    if constexpr (MQ) {
      const int i = (b % n_cg) * tpg + c / g_heads;
      return ((long long)(b / n_cg) * n_q + i) * num_q_heads + (long long)j * g_heads + c % g_heads;
    }
    return row0 + c;
  };
  if (n == 0) {
    if constexpr (MQ) {
      for (int e = tid; e < cols * D; e += blockDim.x) out[out_row(e / D) * D + e % D] = 0.0f;
    } else {
      for (int e = tid; e < group * D; e += blockDim.x) out[row0 * D + e] = 0.0f;
    }
    return;
  }
  if (usl.first == usl.last) return;
  // this thread's quads: four channels of one column each, quads tid,
  // tid + kCombineThreads, ... of the unit's cols * D / 4 (at most 256)
  constexpr int kQ = (256 + kCombineThreads - 1) / kCombineThreads;
  const int nquad = cols * D / 4;
  if (tid >= nquad) return;
  int e0[kQ], hq[kQ];
  bool act[kQ];
  float M[kQ], W[kQ], A[kQ][4];
#pragma unroll
  for (int x = 0; x < kQ; ++x) {
    const int qd = tid + x * kCombineThreads;
    act[x] = qd < nquad;
    e0[x] = act[x] ? qd * 4 : 0;
    hq[x] = e0[x] / D;
    M[x] = -INFINITY;
    W[x] = 0.0f;
    A[x][0] = A[x][1] = A[x][2] = A[x][3] = 0.0f;
  }
  for (long long s0 = usl.first; s0 <= usl.last; s0 += kMaxSl) {
    const int cnt = (int)min((long long)kMaxSl, usl.last - s0 + 1);
    // slices of this round holding a partial (block-uniform)
    unsigned long long mask = mask0;
    if (s0 != usl.first) {
      mask = 0;
      for (int i = 0; i < cnt; ++i)
        if (usl.has_part(s0 + i)) mask |= 1ull << i;
    }
    // one round of loads: lse and the quads of kBatch partials
    constexpr int kBatch = 4;
    for (int i0 = 0; i0 < cnt; i0 += kBatch) {
      float l[kQ][kBatch];
      float4 o[kQ][kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int i = i0 + k;
        const bool has = i < cnt && ((mask >> i) & 1);
        const long long slot = s0 + i + u;
#pragma unroll
        for (int x = 0; x < kQ; ++x) {
          l[x][k] = -INFINITY;
          o[x][k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (has && act[x]) {
            l[x][k] = __ldcg(part_lse + slot * group + hq[x]);
            o[x][k] = __ldcg(reinterpret_cast<const float4*>(part_o + slot * group * D + e0[x]));
          }
        }
      }
#pragma unroll
      for (int x = 0; x < kQ; ++x)
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (l[x][k] == -INFINITY) continue;
          const float Mn = fmaxf(M[x], l[x][k]);
          const float a = M[x] == -INFINITY ? 0.0f : exp2f(M[x] - Mn), w = exp2f(l[x][k] - Mn);
          W[x] = W[x] * a + w;
          A[x][0] = A[x][0] * a + w * o[x][k].x;
          A[x][1] = A[x][1] * a + w * o[x][k].y;
          A[x][2] = A[x][2] * a + w * o[x][k].z;
          A[x][3] = A[x][3] * a + w * o[x][k].w;
          M[x] = Mn;
        }
    }
  }
#pragma unroll
  for (int x = 0; x < kQ; ++x) {
    if (!act[x]) continue;
    const float inv = W[x] > 0.0f ? 1.0f / W[x] : 0.0f;
    const int h = hq[x];
    float* dst = MQ ? out + out_row(h) * D + (e0[x] - h * D) : out + row0 * D + e0[x];
    *reinterpret_cast<float4*>(dst) = make_float4(A[x][0] * inv, A[x][1] * inv, A[x][2] * inv, A[x][3] * inv);
  }
}

template <int KV, int D, int BS, int G, int NS, bool TC, bool MQ = false, bool AP = false>
cudaError_t launch_t(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t stream) {
  using SM = Smem<KV, D, BS, G, NS, consumer_warps<KV, TC, BS>(), TC>;
  auto kern = paged_gqa_decode_kernel<KV, D, BS, G, NS, TC, MQ, AP>;
  static std::atomic<unsigned long long> ready_dec{0}, ready_comb{0};  // per instantiation, per device
  cudaError_t e = prepare_kernel(kern, (int)SM::kBytes, ready_dec);
  if (e != cudaSuccess) return e;
  e = prepare_kernel(splitkv_combine_kernel<D, MQ>, 0, ready_comb);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.num_ctas);
  cfg.blockDim = dim3((consumer_warps<KV, TC, BS>() + 2) * 32);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return e;
  const int units = prm.batch * prm.pool.num_kv_heads;
  if (units == 0 || prm.fused) return cudaSuccess;
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<D, MQ>, prm.seq_lens, (const int32_t*)prm.pre_cost,
                            (const float*)prm.part_o, (const float*)prm.part_lse, prm.out, prm.batch,
                            prm.pool.num_kv_heads, prm.group, prm.num_q_heads, L.num_ctas, prm.pool.block_size,
                            prm.max_blocks, prm.unit_cost, prm.early_plan, prm.n_q, prm.n_cg, prm.tpg,
                            prm.g_heads);
}

// Stages per consumer warp: as many pages in flight as the shared memory
// allows next to the fixed parts (1..8 per warp, largest that fits with 1 KB
// of static shared memory to spare). Bytes in flight per SM are what sustains
// HBM bandwidth (Little's law), so the ring gets the rest.
template <int KV, int D, int BS, int G, int W, bool TC, int N>
constexpr int largest_ring() {
  if constexpr (N <= 1) {
    return 1;
  } else if constexpr (Smem<KV, D, BS, G, N, W, TC>::kBytes + 1024 <= 227 * 1024) {
    return N;
  } else {
    return largest_ring<KV, D, BS, G, W, TC, N - 1>();
  }
}

template <int KV, int D, int BS, int G, int W, bool TC>
constexpr int stages_per_warp() {
  return largest_ring<KV, D, BS, G, W, TC, 8>();
}

template <int KV, int D, int BS, bool TC>
cudaError_t dispatch_g(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t s) {
  constexpr int W = consumer_warps<KV, TC, BS>();
  // several query tokens per sequence: column groups of up to 8 columns
  if (L.n_q > 1) return launch_t<KV, D, BS, 8, stages_per_warp<KV, D, BS, 8, W, TC>(), TC, true>(prm, L, s);
  if (prm.append) {  // the fused decode step
    if (L.group <= 2) return launch_t<KV, D, BS, 2, stages_per_warp<KV, D, BS, 2, W, TC>(), TC, false, true>(prm, L, s);
    if (L.group <= 4) return launch_t<KV, D, BS, 4, stages_per_warp<KV, D, BS, 4, W, TC>(), TC, false, true>(prm, L, s);
    return launch_t<KV, D, BS, 8, stages_per_warp<KV, D, BS, 8, W, TC>(), TC, false, true>(prm, L, s);
  }
  if (L.group <= 2) return launch_t<KV, D, BS, 2, stages_per_warp<KV, D, BS, 2, W, TC>(), TC>(prm, L, s);
  if (L.group <= 4) return launch_t<KV, D, BS, 4, stages_per_warp<KV, D, BS, 4, W, TC>(), TC>(prm, L, s);
  return launch_t<KV, D, BS, 8, stages_per_warp<KV, D, BS, 8, W, TC>(), TC>(prm, L, s);
}

template <int KV, int D, int BS>
cudaError_t dispatch_path(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t s) {
  if constexpr (KV == PA_KV_BF16 || D == 128) {
    if (L.tensor_cores) return dispatch_g<KV, D, BS, true>(prm, L, s);
  }
  return dispatch_g<KV, D, BS, false>(prm, L, s);
}

template <int KV>
cudaError_t dispatch_kv(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t s) {
  const int D = prm.pool.head_dim, BS = prm.pool.block_size;
  if (D == 64 && BS == 16) return dispatch_path<KV, 64, 16>(prm, L, s);
  if (D == 64 && BS == 32) return dispatch_path<KV, 64, 32>(prm, L, s);
  if (D == 128 && BS == 16) return dispatch_path<KV, 128, 16>(prm, L, s);
  if (D == 128 && BS == 32) return dispatch_path<KV, 128, 32>(prm, L, s);
  return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

template <int KV, int D, int BS, bool TC>
size_t smem_bytes_g(int group) {
  constexpr int W = consumer_warps<KV, TC, BS>();
  constexpr int N2 = stages_per_warp<KV, D, BS, 2, W, TC>();
  constexpr int N4 = stages_per_warp<KV, D, BS, 4, W, TC>();
  constexpr int N8 = stages_per_warp<KV, D, BS, 8, W, TC>();
  static_assert(Smem<KV, D, BS, 8, N8, W, TC>::kBytes <= 227 * 1024, "shared memory budget");
  if (group <= 2) return Smem<KV, D, BS, 2, N2, W, TC>::kBytes;
  if (group <= 4) return Smem<KV, D, BS, 4, N4, W, TC>::kBytes;
  return Smem<KV, D, BS, 8, N8, W, TC>::kBytes;
}

template <int KV, bool TC>
size_t smem_bytes_kv(int D, int BS, int group) {
  if (D == 64 && BS == 16) return smem_bytes_g<KV, 64, 16, TC>(group);
  if (D == 64 && BS == 32) return smem_bytes_g<KV, 64, 32, TC>(group);
  if (D == 128 && BS == 16) return smem_bytes_g<KV, 128, 16, TC>(group);
  return smem_bytes_g<KV, 128, 32, TC>(group);
}

// Carve the workspace and launch decode + combine for pools of format KV.
template <int KV>
cudaError_t launch_decode_kv(const PoolDev& pool, const PoolMaps& maps, const void* q,
                             const int32_t* block_table, const int32_t* seq_lens, float* out,
                             void* workspace, DecodeLaunch& L, cudaStream_t stream) {
  const size_t slots = (size_t)L.num_ctas + (size_t)L.batch * pool.num_kv_heads;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned long long* tickets = reinterpret_cast<unsigned long long*>(ws);
  ws += align256(sizeof(unsigned long long) * (size_t)L.batch * pool.num_kv_heads);
  L.pre_cost = reinterpret_cast<int32_t*>(ws);
  ws += align256(sizeof(int32_t) * ((size_t)L.batch + 1));
  L.part_lse = reinterpret_cast<float*>(ws);
  ws += align256(sizeof(float) * slots * L.group);
  L.part_o = reinterpret_cast<float*>(ws);
  DecodeParams prm;
  prm.maps = maps;
  prm.pool = pool;
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.out = out;
  prm.pre_cost = L.pre_cost;
  prm.unit_cost = L.unit_cost;
  prm.part_o = L.part_o;
  prm.part_lse = L.part_lse;
  prm.tickets = tickets;
  prm.epoch = L.epoch;
  prm.fused = L.fused_combine && L.n_q <= 1 ? 1 : 0;  // no in-kernel merge of column groups
  prm.early_plan = L.early_plan ? 1 : 0;
  prm.batch = L.batch;
  prm.num_q_heads = L.num_q_heads;
  prm.group = L.group;
  prm.max_blocks = L.max_blocks;
  prm.scale_log2 = L.scale_log2;
  prm.n_q = L.n_q > 1 ? L.n_q : 1;
  prm.n_cg = L.n_q > 1 ? L.n_cg : 1;
  prm.tpg = L.n_q > 1 ? L.tpg : 1;
  prm.g_heads = L.n_q > 1 ? L.g_heads : L.group;
  prm.k_new = static_cast<const __nv_bfloat16*>(L.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(L.v_new);
  prm.append = (L.n_q <= 1 && L.k_new != nullptr && L.v_new != nullptr) ? 1 : 0;
  return dispatch_kv<KV>(prm, L, stream);
}

}  // namespace

}  // namespace pa
