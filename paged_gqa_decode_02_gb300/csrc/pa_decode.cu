// paged_gqa_decode + splitkv_combine for GB300 (sm_103a).
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
// heads of its group. The units' blocks are concatenated in (b, j, block)
// order into one list of T pages; thread block i of G takes the contiguous
// slice [i*T/G, (i+1)*T/G). Every SM therefore streams the same number of
// bytes whatever the length mix. A unit that lies inside one slice is
// written straight to `out`; a unit cut by slice boundaries leaves one
// partial (o = acc / l, lse = m + log2 l) per slice, merged by the combine
// kernel with log-sum-exp weights.
//
// Inside a thread block: warp 0 is the producer. It reads block-table entries
// 32 at a time and issues 1-D TMA bulk copies (cp.async.bulk) of each page's
// K and V (plus scales / zero points) into a ring of shared-memory stages,
// one sub-ring per consumer warp, completing on mbarriers. Consumer warps
// take pages round-robin, keep a private online-softmax state per unit
// (fp32, max/sum reductions with warp shuffles), and merge their states
// through shared memory at the end of each unit.
//
// Every wait is bounded: on expiry the thread block records
// PA_DEVERR_TIMEOUT, stops waiting and computing, keeps the barrier sequence
// (so no thread is stranded) and drains its outstanding copies before exit.
#include <float.h>

#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSegs = 64;

// One contiguous run of pages of one unit inside a thread block's slice.
struct Seg {
  int32_t b, h;      // sequence, kv head
  int32_t lp0;       // first logical block of the run
  int32_t npages;    // pages in the run
  int32_t k0;        // index of the run's first page within the slice
  int32_t len;       // sequence length (tokens)
  int32_t slot;      // partial slot (cta + unit), or -1 when written directly
  int32_t pad;
};

template <int KV, int D, int BS>
struct PageGeom {
  static constexpr int kElemBits = KV == PA_KV_BF16 ? 16 : (KV == PA_KV_UINT8 ? 8 : 4);
  static constexpr int kPageBytes = BS * D * kElemBits / 8;      // one of K or V
  static constexpr int kMetaBytes = KV == PA_KV_BF16 ? 0 : D * 4;  // one of scale or zp
  static constexpr int kStageBytes = 2 * kPageBytes + 4 * kMetaBytes;
  // offsets inside a stage
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kPageBytes;
  static constexpr int kOffKs = 2 * kPageBytes;
  static constexpr int kOffKz = kOffKs + kMetaBytes;
  static constexpr int kOffVs = kOffKz + kMetaBytes;
  static constexpr int kOffVz = kOffVs + kMetaBytes;
};

template <int KV, int D, int BS, int G, int NS>
struct Smem {
  using PG = PageGeom<KV, D, BS>;
  static constexpr int kStages = kConsumerWarps * NS;
  static constexpr int kQBytes = G * D * 2;
  static constexpr size_t kOffBars = 0;  // full[kStages], empty[kStages], qfull[2], qempty[2]
  static constexpr size_t kBarBytes = (2 * kStages + 4) * 8;
  static constexpr size_t kOffFlags = kBarBytes;  // int32 per stage
  static constexpr size_t kOffSegs = (kOffFlags + kStages * 4 + 15) / 16 * 16;
  static constexpr size_t kOffPlan = kOffSegs + kMaxSegs * sizeof(Seg);  // 32 int64
  static constexpr size_t kOffQ = (kOffPlan + 32 * 8 + 127) / 128 * 128;
  static constexpr size_t kOffStash = kOffQ + 2 * kQBytes;
  static constexpr size_t kStashAccBytes = (size_t)kConsumerWarps * G * D * 4;
  static constexpr size_t kOffStashML = kOffStash + kStashAccBytes;
  static constexpr size_t kOffPbuf = kOffStashML + kConsumerWarps * G * 2 * 4;
  static constexpr size_t kPbufBytes = (size_t)kConsumerWarps * BS * G * 4;
  static constexpr size_t kOffStages = (kOffPbuf + kPbufBytes + 127) / 128 * 128;
  static constexpr size_t kBytes = kOffStages + (size_t)kStages * PG::kStageBytes;
};

struct DecodeParams {
  PoolDev pool;
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* out;
  int32_t* pre_pages;
  float* part_o;
  float* part_lse;
  int batch;
  int num_q_heads;
  int group;
  int max_blocks;
  float scale_log2;
};

// Sequence length clamped to what the table can hold; bad lengths count as 0.
__device__ __forceinline__ int seq_len_checked(const DecodeParams& p, int b, bool report) {
  const int len = p.seq_lens[b];
  if (len < 0 || (long long)len > (long long)p.max_blocks * p.pool.block_size) {
    if (report) set_error(p.pool.err, PA_DEVERR_SEQ_LEN);
    return 0;
  }
  return len;
}

// first / last thread block whose slice contains flattened page x
__device__ __forceinline__ long long owner_of(long long x, long long T, long long G) {
  return ((x + 1) * G - 1) / T;
}

// Block-wide inclusive scan of one int per thread (all kThreads threads call).
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
  for (int w = 0; w < kThreads / 32; ++w) {
    const int t = warp_tot[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return x + before;
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

  __device__ __forceinline__ void page(const uint8_t* stage, int valid, float* pbuf) {
    const int lane = threadIdx.x & 31;
    const uint8_t* kp = stage + PG::kOffK;
    const uint8_t* vp = stage + PG::kOffV;
    float ksc[CPL], vsc[CPL];
    int32_t kzp[CPL], vzp[CPL];
    if (KV != PA_KV_BF16) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        ksc[c] = reinterpret_cast<const float*>(stage + PG::kOffKs)[lane * CPL + c];
        kzp[c] = reinterpret_cast<const int32_t*>(stage + PG::kOffKz)[lane * CPL + c];
        vsc[c] = reinterpret_cast<const float*>(stage + PG::kOffVs)[lane * CPL + c];
        vzp[c] = reinterpret_cast<const int32_t*>(stage + PG::kOffVz)[lane * CPL + c];
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
      s[ch] = t < valid ? part[0] : -INFINITY;
    }
    // ---- online softmax (head lane % G)
    float pmax = s[0];
#pragma unroll
    for (int ch = 1; ch < NCH; ++ch) pmax = fmaxf(pmax, s[ch]);
#pragma unroll
    for (int off = G; off < 32; off <<= 1) pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, off));
    const float m_new = fmaxf(m_run, pmax);
    const float alpha = exp2f(m_run - m_new);
    float psum = 0.0f;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
      const float p = exp2f(s[ch] - m_new);
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
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int c = 0; c < CPL; ++c) st_acc[h * D + lane * CPL + c] = acc[h][c];
  }
};

// ------------------------------------------------------------------ the decode kernel
template <int KV, int D, int BS, int G, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    paged_gqa_decode_kernel(const DecodeParams p) {
  using SM = Smem<KV, D, BS, G, NS>;
  using PG = PageGeom<KV, D, BS>;
  constexpr int NST = SM::kStages;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kOffBars);
  uint64_t* empty = full + NST;
  uint64_t* qfull = empty + NST;
  uint64_t* qempty = qfull + 2;
  int32_t* stage_flag = reinterpret_cast<int32_t*>(smem + SM::kOffFlags);
  Seg* segs = reinterpret_cast<Seg*>(smem + SM::kOffSegs);
  long long* plan = reinterpret_cast<long long*>(smem + SM::kOffPlan);
  uint8_t* qslots = smem + SM::kOffQ;
  float* stash_acc = reinterpret_cast<float*>(smem + SM::kOffStash);
  float* stash_ml = reinterpret_cast<float*>(smem + SM::kOffStashML);
  float* pbuf_all = reinterpret_cast<float*>(smem + SM::kOffPbuf);
  uint8_t* stages = smem + SM::kOffStages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.pool.num_kv_heads;
  const int g = p.group;
  const long long Gc = gridDim.x, cta = blockIdx.x;
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int abort_flag;
  __shared__ int issued_n[NST];  // last fill issued per stage (drain on abort)
  __shared__ int q_issued[2];    // last q segment index issued per slot

  // Launched with programmatic stream serialization: let the combine kernel
  // be scheduled early, but touch no global memory before the preceding
  // kernel in the stream has completed.
  pdl_launch_dependents();
  pdl_wait();

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
    abort_flag = 0;
    q_issued[0] = q_issued[1] = -1;
    fence_mbar_init();
  }

  // ---- plan: total pages, this slice, and where it starts
  long long npages_all = 0;
  {
    int part = 0;
    for (int b = tid; b < p.batch; b += kThreads) part += (seq_len_checked(p, b, cta == 0) + BS - 1) / BS;
    int tot;
    block_incl_scan(part, warp_tot, tot);
    npages_all = tot;
  }
  const long long T = npages_all * Hkv;
  const long long s_i = T * cta / Gc, e_i = T * (cta + 1) / Gc;
  // CTA 0 publishes the per-sequence prefix for the combine kernel; every
  // CTA finds the sequence holding its first page.
  if (tid == 0) plan[0] = -1;
  {
    int running = 0;
    for (int base = 0; base < p.batch; base += kThreads) {
      const int b = base + tid;
      const int n = b < p.batch ? (seq_len_checked(p, b, false) + BS - 1) / BS : 0;
      int tot;
      const int incl = block_incl_scan(n, warp_tot, tot);
      const long long lo = (long long)(running + incl - n) * Hkv;
      const long long hi = (long long)(running + incl) * Hkv;
      if (cta == 0 && b < p.batch) {
        p.pre_pages[b] = running + incl - n;
        if (b == p.batch - 1) p.pre_pages[p.batch] = running + incl;
      }
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
    if (cta == 0 && p.batch == 0 && tid == 0) p.pre_pages[0] = 0;
  }
  __syncthreads();
  if (s_i >= e_i) return;  // no pages for this thread block

  long long cur_b = plan[0], cur_base = plan[1];  // sequence holding `pos` and its first page
  long long pos = s_i;
  int seg_counter = 0;      // segments started so far (q slot ring index)
  uint64_t pol = policy_evict_first();

  while (pos < e_i) {
    // ---- build this window's segment list (warp 0)
    if (warp == 0) {
      int nseg = 0;
      long long b0 = cur_b, base0 = cur_base, wpos = pos;
      bool done = false;
      while (!done && b0 < p.batch) {
        const long long bb = b0 + lane;
        const int len = bb < p.batch ? seq_len_checked(p, (int)bb, false) : 0;
        const int n = (len + BS - 1) / BS;
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        const long long my_base = base0 + (long long)(x - n) * Hkv;
        const long long my_end = my_base + (long long)n * Hkv;
        const bool overl = n > 0 && my_end > wpos && my_base < e_i && bb < p.batch;
        unsigned mask = __ballot_sync(0xffffffffu, overl);
        while (mask) {
          const int src = __ffs(mask) - 1;
          mask &= mask - 1;
          const long long sb = b0 + src;
          const long long sbase = __shfl_sync(0xffffffffu, my_base, src);
          const int sn = __shfl_sync(0xffffffffu, n, src);
          const int slen = __shfl_sync(0xffffffffu, len, src);
          const int h_lo = (int)max(0LL, (wpos - sbase) / sn);
          const int h_hi = (int)min((long long)Hkv - 1, (e_i - 1 - sbase) / sn);
          for (int h = h_lo; h <= h_hi && !done; ++h) {
            const long long us = sbase + (long long)h * sn, ue = us + sn;
            const long long lo = max(us, wpos), hi = min(ue, e_i);
            if (lo >= hi) continue;
            if (lane == 0) {
              Seg sg;
              sg.b = (int)sb;
              sg.h = h;
              sg.lp0 = (int)(lo - us);
              sg.npages = (int)(hi - lo);
              sg.k0 = (int)(lo - s_i);
              sg.len = slen;
              const long long first = owner_of(us, T, Gc), last = owner_of(ue - 1, T, Gc);
              sg.slot = first == last ? -1 : (int)(cta + sb * Hkv + h);
              sg.pad = 0;
              segs[nseg] = sg;
            }
            ++nseg;
            wpos = hi;
            if (hi >= e_i) done = true;
            if (nseg == kMaxSegs && !done) {
              done = true;
              // resume at the sequence holding wpos
              if (wpos >= sbase + (long long)sn * Hkv) {
                cur_b = sb + 1;
                cur_base = sbase + (long long)sn * Hkv;
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
      }
    }
    __syncthreads();
    const int nseg = (int)plan[2];
    const long long wend = plan[3];
    cur_b = plan[4];
    cur_base = plan[5];
    const int kw0 = (int)(pos - s_i), kw1 = (int)(wend - s_i);

    if (warp == 0) {
      // ---------------------------------------------------------- producer
      int si = 0;  // segment of the current page
      int qseg = 0;
      for (int kb = kw0; kb < kw1; kb += 32) {
        const int my_k = kb + lane;
        int my_phys = -1;
        if (my_k < kw1) {
          int s = 0;
          while (s + 1 < nseg && my_k >= segs[s + 1].k0) ++s;
          const Seg& sg = segs[s];
          my_phys = p.block_table[(long long)sg.b * p.max_blocks + sg.lp0 + (my_k - sg.k0)];
        }
        const int cnt = min(32, kw1 - kb);
        for (int j = 0; j < cnt; ++j) {
          const int k = kb + j;
          const int phys = __shfl_sync(0xffffffffu, my_phys, j);
          while (si + 1 < nseg && k >= segs[si + 1].k0) ++si;
          if (lane == 0) {
            const Seg& sg = segs[si];
            const bool aborted = abort_flag != 0;
            // q of a unit goes out with its first page in this slice
            while (qseg <= si) {
              const int gs = seg_counter + qseg;
              const int slot = gs & 1;
              bool ok = true;
              if (gs >= 2 && !aborted) ok = mbar_wait_bounded(&qempty[slot], ((gs >> 1) - 1) & 1);
              if (!ok) {
                set_error(p.pool.err, PA_DEVERR_TIMEOUT);
                abort_flag = 1;
              }
              const Seg& qs = segs[qseg];
              const uint16_t* qsrc = p.q + ((long long)qs.b * p.num_q_heads + (long long)qs.h * g) * D;
              if (abort_flag) {
                mbar_arrive(&qfull[slot]);
              } else {
                q_issued[slot] = gs;
                mbar_arrive_expect_tx(&qfull[slot], g * D * 2);
                bulk_g2s(qslots + slot * SM::kQBytes, qsrc, g * D * 2, &qfull[slot], pol);
              }
              ++qseg;
            }
            const int stage = k % NST;
            const int n = k / NST;
            bool ok = true;
            if (n >= 1 && !abort_flag) ok = mbar_wait_bounded(&empty[stage], (n - 1) & 1);
            if (!ok) {
              set_error(p.pool.err, PA_DEVERR_TIMEOUT);
              abort_flag = 1;
            }
            if (phys < 0 || phys >= p.pool.num_blocks || abort_flag) {
              if (!abort_flag) set_error(p.pool.err, PA_DEVERR_BLOCK_TABLE);
              stage_flag[stage] = 1;
              mbar_arrive(&full[stage]);
            } else {
              stage_flag[stage] = 0;
              uint8_t* dst = stages + (size_t)stage * PG::kStageBytes;
              const long long page = (long long)phys * Hkv + sg.h;
              issued_n[stage] = n;
              mbar_arrive_expect_tx(&full[stage], PG::kStageBytes);
              bulk_g2s(dst + PG::kOffK, p.pool.k + page * PG::kPageBytes, PG::kPageBytes, &full[stage], pol);
              bulk_g2s(dst + PG::kOffV, p.pool.v + page * PG::kPageBytes, PG::kPageBytes, &full[stage], pol);
              if (KV != PA_KV_BF16) {
                bulk_g2s(dst + PG::kOffKs, p.pool.k_scale + page * D, PG::kMetaBytes, &full[stage], pol);
                bulk_g2s(dst + PG::kOffKz, p.pool.k_zp + page * D, PG::kMetaBytes, &full[stage], pol);
                bulk_g2s(dst + PG::kOffVs, p.pool.v_scale + page * D, PG::kMetaBytes, &full[stage], pol);
                bulk_g2s(dst + PG::kOffVz, p.pool.v_zp + page * D, PG::kMetaBytes, &full[stage], pol);
              }
            }
          }
          __syncwarp();
        }
      }
      // units without pages in this window never happen: every segment has >= 1 page
    } else {
      // ---------------------------------------------------------- consumers
      const int cw = warp - 1;
      float* pbuf = pbuf_all + cw * BS * G;
      FmaConsumer<KV, D, BS, G> cons;
      for (int si = 0; si < nseg; ++si) {
        const Seg sg = segs[si];
        const int gs = seg_counter + si;
        const int slot = gs & 1;
        bool ok = abort_flag == 0 && mbar_wait_bounded(&qfull[slot], (gs >> 1) & 1);
        if (!ok && abort_flag == 0) {
          if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
          abort_flag = 1;
        }
        cons.begin_unit(reinterpret_cast<const uint16_t*>(qslots + slot * SM::kQBytes), g, p.scale_log2);
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[slot]);
        // my pages: k = k0 + i with k % W == cw
        const int kfirst = sg.k0 + ((cw - sg.k0 % kConsumerWarps) + kConsumerWarps) % kConsumerWarps;
        for (int k = kfirst; k < sg.k0 + sg.npages; k += kConsumerWarps) {
          const int stage = k % NST;
          const int n = k / NST;
          bool okp = abort_flag == 0 && mbar_wait_bounded(&full[stage], n & 1);
          if (!okp && abort_flag == 0) {
            if (lane == 0) set_error(p.pool.err, PA_DEVERR_TIMEOUT);
            abort_flag = 1;
          }
          if (okp && stage_flag[stage] == 0) {
            const int lp = sg.lp0 + (k - sg.k0);
            const int valid = min(BS, sg.len - lp * BS);
            cons.page(stages + (size_t)stage * PG::kStageBytes, valid, pbuf);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        }
        cons.deposit(stash_acc + cw * G * D, stash_ml + cw * G * 2);
        named_bar_sync(1, kConsumerWarps * 32);
        // ---- merge the warps' states and write
        const int ctid = tid - 32;
        const long long row0 = (long long)sg.b * p.num_q_heads + (long long)sg.h * g;
        for (int e = ctid; e < g * D; e += kConsumerWarps * 32) {
          const int h = e / D, c = e % D;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, stash_ml[(w * G + h) * 2]);
          float Lsum = 0.0f, A = 0.0f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = stash_ml[(w * G + h) * 2];
            const float f = mw == -INFINITY ? 0.0f : exp2f(mw - M);
            Lsum += stash_ml[(w * G + h) * 2 + 1] * f;
            A += stash_acc[(w * G + h) * D + c] * f;
          }
          const float o = Lsum > 0.0f ? A / Lsum : 0.0f;
          if (sg.slot < 0) {
            p.out[(row0 + h) * D + c] = o;
          } else {
            p.part_o[((long long)sg.slot * g + h) * D + c] = o;
            if (c == 0) p.part_lse[(long long)sg.slot * g + h] = Lsum > 0.0f ? M + log2f(Lsum) : -INFINITY;
          }
        }
        named_bar_sync(1, kConsumerWarps * 32);
      }
    }
    seg_counter += nseg;
    pos = wend;
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
template <int D>
__global__ void __launch_bounds__(128)
    splitkv_combine_kernel(const int32_t* pre_pages, const float* part_o, const float* part_lse,
                           float* out, int batch, int num_kv_heads, int group, int num_q_heads,
                           int num_ctas) {
  pdl_launch_dependents();
  pdl_wait();
  const int u = blockIdx.x;
  const int b = u / num_kv_heads, j = u % num_kv_heads;
  const long long pre = pre_pages[b];
  const long long n = pre_pages[b + 1] - pre;
  const long long T = (long long)pre_pages[batch] * num_kv_heads;
  const long long row0 = (long long)b * num_q_heads + (long long)j * group;
  if (n == 0) {
    for (int e = threadIdx.x; e < group * D; e += blockDim.x) out[row0 * D + e] = 0.0f;
    return;
  }
  const long long us = pre * num_kv_heads + (long long)j * n;
  const long long first = owner_of(us, T, num_ctas), last = owner_of(us + n - 1, T, num_ctas);
  if (first == last) return;
  // slice i holds a partial of this unit (in slot i + u) iff its page range
  // meets the unit's; slices between first and last can be empty when there
  // are more slices than pages
  auto has_part = [&](long long i) {
    const long long a = T * i / num_ctas, z = T * (i + 1) / num_ctas;
    return (a > us ? a : us) < (z < us + n ? z : us + n);
  };
  for (int e = threadIdx.x; e < group * D; e += blockDim.x) {
    const int h = e / D, c = e % D;
    float M = -INFINITY;
    for (long long i = first; i <= last; ++i)
      if (has_part(i)) M = fmaxf(M, part_lse[(i + u) * group + h]);
    float W = 0.0f, A = 0.0f;
    for (long long i = first; i <= last; ++i) {
      if (!has_part(i)) continue;
      const long long s = i + u;
      const float l = part_lse[s * group + h];
      const float w = l == -INFINITY ? 0.0f : exp2f(l - M);
      W += w;
      A += w * part_o[(s * group + h) * D + c];
    }
    out[(row0 + h) * D + c] = W > 0.0f ? A / W : 0.0f;
  }
}

template <int KV, int D, int BS, int G, int NS>
cudaError_t launch_t(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t stream) {
  using SM = Smem<KV, D, BS, G, NS>;
  auto kern = paged_gqa_decode_kernel<KV, D, BS, G, NS>;
  static bool attr_set = false;  // per instantiation; set before first launch
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::kBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SM::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm);
  if (e != cudaSuccess) return e;
  const int units = prm.batch * prm.pool.num_kv_heads;
  if (units == 0) return cudaSuccess;
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<D>, (const int32_t*)prm.pre_pages,
                            (const float*)prm.part_o, (const float*)prm.part_lse, prm.out,
                            prm.batch, prm.pool.num_kv_heads, prm.group, prm.num_q_heads,
                            L.num_ctas);
}

// Stages per consumer warp: as many pages in flight as fit a ~160 KB ring
// (2..4 per warp).
template <int KV, int D, int BS>
constexpr int stages_per_warp() {
  constexpr int n = (160 * 1024) / (kConsumerWarps * PageGeom<KV, D, BS>::kStageBytes);
  return n < 2 ? 2 : (n > 4 ? 4 : n);
}

template <int KV, int D, int BS>
cudaError_t dispatch_g(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t s) {
  constexpr int NS = stages_per_warp<KV, D, BS>();
  if (L.group <= 2) return launch_t<KV, D, BS, 2, NS>(prm, L, s);
  if (L.group <= 4) return launch_t<KV, D, BS, 4, NS>(prm, L, s);
  return launch_t<KV, D, BS, 8, NS>(prm, L, s);
}

template <int KV>
cudaError_t dispatch_kv(const DecodeParams& prm, const DecodeLaunch& L, cudaStream_t s) {
  const int D = prm.pool.head_dim, BS = prm.pool.block_size;
  if (D == 64 && BS == 16) return dispatch_g<KV, 64, 16>(prm, L, s);
  if (D == 64 && BS == 32) return dispatch_g<KV, 64, 32>(prm, L, s);
  if (D == 128 && BS == 16) return dispatch_g<KV, 128, 16>(prm, L, s);
  if (D == 128 && BS == 32) return dispatch_g<KV, 128, 32>(prm, L, s);
  return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

template <int KV, int D, int BS>
size_t smem_bytes_g(int group) {
  constexpr int NS = stages_per_warp<KV, D, BS>();
  static_assert(Smem<KV, D, BS, 8, NS>::kBytes <= 227 * 1024, "shared memory budget");
  if (group <= 2) return Smem<KV, D, BS, 2, NS>::kBytes;
  if (group <= 4) return Smem<KV, D, BS, 4, NS>::kBytes;
  return Smem<KV, D, BS, 8, NS>::kBytes;
}

template <int KV>
size_t smem_bytes_kv(int D, int BS, int group) {
  if (D == 64 && BS == 16) return smem_bytes_g<KV, 64, 16>(group);
  if (D == 64 && BS == 32) return smem_bytes_g<KV, 64, 32>(group);
  if (D == 128 && BS == 16) return smem_bytes_g<KV, 128, 16>(group);
  return smem_bytes_g<KV, 128, 32>(group);
}

}  // namespace

size_t decode_workspace_bytes(int num_ctas, int batch, int num_kv_heads, int group, int head_dim) {
  const size_t slots = (size_t)num_ctas + (size_t)batch * num_kv_heads;
  return align256(sizeof(int32_t) * ((size_t)batch + 1)) + align256(sizeof(float) * slots * group) +
         align256(sizeof(float) * slots * group * head_dim);
}

int decode_ctas_per_sm(int kv_dtype, int block_size, int head_dim, int group) {
  size_t smem = kv_dtype == PA_KV_BF16    ? smem_bytes_kv<PA_KV_BF16>(head_dim, block_size, group)
                : kv_dtype == PA_KV_UINT8 ? smem_bytes_kv<PA_KV_UINT8>(head_dim, block_size, group)
                                          : smem_bytes_kv<PA_KV_UINT4>(head_dim, block_size, group);
  const size_t per_sm = 227 * 1024;
  int n = (int)(per_sm / (smem + 1024));
  return n < 1 ? 1 : (n > 4 ? 4 : n);
}

cudaError_t launch_decode(int kv_dtype, const PoolDev& pool, const void* q,
                          const int32_t* block_table, const int32_t* seq_lens, float* out,
                          void* workspace, DecodeLaunch& L, cudaStream_t stream) {
  const size_t slots = (size_t)L.num_ctas + (size_t)L.batch * pool.num_kv_heads;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  L.pre_pages = reinterpret_cast<int32_t*>(ws);
  ws += align256(sizeof(int32_t) * ((size_t)L.batch + 1));
  L.part_lse = reinterpret_cast<float*>(ws);
  ws += align256(sizeof(float) * slots * L.group);
  L.part_o = reinterpret_cast<float*>(ws);
  DecodeParams prm;
  prm.pool = pool;
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.out = out;
  prm.pre_pages = L.pre_pages;
  prm.part_o = L.part_o;
  prm.part_lse = L.part_lse;
  prm.batch = L.batch;
  prm.num_q_heads = L.num_q_heads;
  prm.group = L.group;
  prm.max_blocks = L.max_blocks;
  prm.scale_log2 = L.scale_log2;
  if (kv_dtype == PA_KV_BF16) return dispatch_kv<PA_KV_BF16>(prm, L, stream);
  if (kv_dtype == PA_KV_UINT8) return dispatch_kv<PA_KV_UINT8>(prm, L, stream);
  if (kv_dtype == PA_KV_UINT4) return dispatch_kv<PA_KV_UINT4>(prm, L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
