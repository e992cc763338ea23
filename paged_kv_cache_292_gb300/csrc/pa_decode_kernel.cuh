// Paged decode attention for sm_103a.
//
// What it computes is section 3.2 ("内核执行流程（简化版）") of "vLLM
// three-process architecture and the PagedAttention kernel": for each
// sequence, look up its block table (step 1), bound the walk by its valid
// length (step 2), gather K/V from the scattered physical blocks (step 3),
// attend with the step's query (step 4) and write the output (step 5).  The
// same section's "精妙之处" asks for the gather to be planned up front and for
// copies to overlap compute on the GPU's separate copy engine; here that is
// two producer warps driving the TMA engine's copies into a ring of
// shared-memory stages while consumer warps compute on earlier stages.
//
// Kernel 1 (pa_decode_kernel), one CTA per (token range, KV-head group):
//   * The flattened tile list of the batch is cut into equal ranges (see
//     pa_schedule.h), so every CTA moves the same K/V bytes.
//   * The last two warps (the producers) walk the range tile by tile; both
//     follow every tile's bookkeeping and each takes alternate tiles: for a
//     tile of 16 tokens it looks up the block ids and copies K and V into the
//     tile's stage.
//     A token row is the `Hg` KV heads of the CTA's group, contiguous in the pool
//     ([block, slot, head, dim] layout), e.g. 2 KiB for 8 heads x 128 x bf16.
//     Tensor-core paths (bf16, FP8): one tensor-map box per run of
//     gcd(block_size, 16) rows of one block, landing with the 128-byte
//     swizzle in rows of an odd number of 128-byte lines (see RowPtr), so
//     ldmatrix reads of 8 consecutive tokens hit distinct banks.  fp32: one
//     bulk copy per token row, rows `row + 16` bytes apart.  Each sequence's
//     query slice is copied once into a small ring of its own.
//   * Each consumer warp owns one KV head and its G query heads (with several
//     query tokens and more than 8 (query, head) columns, two to four warps
//     share a KV head, 8 columns each).  bf16: S^T[16 tok x 8] = K_tile[16 x D] *
//     Q^T[D x 8] on the tensor cores (mma.sync m16n8k16, query heads padded
//     to 8), online softmax in registers (running max and sum in the exp2
//     domain), then O^T[D x 8] += V^T[D x 16] * P^T[16 x 8], with P^T obtained
//     from the score fragment by movmatrix.  FP8 pools: codes widened to f16
//     (MmaConsumerF8).  fp32: the same on CUDA cores.  FP8 consumers, and bf16
//     ones that share a KV head's columns with other warps, take two tiles of
//     one segment per pass when the ring has four or more stages (tile2).
//   * Appending calls also write the step's new tokens of each sequence: the
//     consumer warps put them into the staged tile and into the pool
//     (append_new_rows).  Not with several consumer warps per KV head, where
//     that code slowed the consumers' tile loop: the host then writes the rows
//     with a separate kernel ahead of the decode.
//   * Every wait is bounded; a wait that runs out sets PA_DEVERR_TIMEOUT, and
//     the producers let the copies they started land before the CTA retires.
//   * A sequence wholly inside the range is written to `out` directly.  A
//     sequence cut by range boundaries leaves one (m, l, O) partial per range
//     and KV head; the warp that writes the last of them (an atomic ticket per
//     sequence and KV head, no waiting) then merges them all by log-sum-exp:
//     out = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i.  The ticket counters
//     are reset by that warp, so the scratch is left zeroed for the next call.
//   * Empty sequences get zero output rows (all their query rows) from the
//     prologue.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>

#include <type_traits>

#include "../../include/pagedattn.h"
#include "pa_device.cuh"
#include "pa_schedule.h"

namespace pa {

constexpr int kMaxGroupHeads = 8;  // KV heads per CTA (one consumer warp each)
constexpr int kMaxQueryGroup = 8;  // query heads per KV head (MMA N extent)
constexpr int kMaxColumns = 32;    // (query, head) columns per KV head: four consumer warps of 8
// Producer warps per CTA.  They share the walk over the range's tiles and
// take alternate tiles for the per-tile work (block lookup, stage wait, arm,
// copies), so two tiles' issue latencies overlap.
constexpr int kProducers = 2;
constexpr int kRowSkew = 16;       // fp32 stages: bytes between staged rows beyond the row itself
constexpr uint32_t kLine = 128;    // tensor-core stages: bytes per swizzled line
constexpr int kMaxRowBytes = 2048;  // bytes of one staged token row (K or V)
constexpr int kMaxRanges = 4096;    // bounds the partial-result scratch

enum : int { kSegBegin = 1, kSegEnd = 2 };

struct StageMeta {
  int seq;     // sequence index
  int tok0;    // first token of the tile within the sequence
  int nvalid;  // valid tokens in the tile (1..16)
  int flags;   // kSegBegin | kSegEnd | (output slot + 1) << 2 | (slot of range r0) << 4
  int r0, r1;  // first and last range touching the sequence (cut sequences only)
  int ctx;     // the sequence's context length (causal limits of several queries)
  int newfirst;  // appending calls: first tile row holding one of the step's new
                 // tokens (rows newfirst .. nvalid-1; their pool rows are in the
                 // stage's row list); -1 when the tile holds none
};

struct DecodeParams {
  CUtensorMap tm_k, tm_v;  // tensor-core paths: 4-D views of the pools (see make_tensor_maps)
  void* out;
  // Appending calls (bf16, at most 8 (query, head) columns per KV head): K/V
  // rows [num_seqs * num_queries, num_kv_heads, head_size] of each sequence's
  // new tokens (row s * Q + i: position c - Q + i), written into the pool by
  // the decode itself; nullptr otherwise.
  const void* k_new;
  const void* v_new;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t* counters;  // [num_seqs][num_kv_heads] merge tickets; zero between calls
  float* part_ml;   // [R][2][H][2]: (m in log2 units, l)
  float* part_o;    // [R][2][H][D]: un-normalised weighted V sums
  int32_t* error_flag;
  int num_seqs, num_heads, num_kv_heads, group, block_size, max_blocks_per_seq;
  int heads_per_cta;    // Hg
  int num_head_groups;  // HG = Hk / Hg
  int num_ranges;       // R
  int num_physical_blocks;
  int stages, q_slots;
  int num_queries;  // query tokens per sequence (1 for plain decode)
  int split;        // consumer warps per KV head: ceil(G * num_queries / 8), 8 columns each
  float v_scale;    // FP8 pools: value of a V code is decode(code) * v_scale (else 1)
  float k_scale;    // FP8 pools: value of a K code is decode(code) * k_scale (else 1)
  uint32_t row_bytes, pitch, q_bytes, stage_bytes;
  uint32_t lines;      // tensor-core stages: 128-byte lines per staged token row
  uint32_t box_rows;   // token rows per tensor copy: gcd(block_size, 16)
  uint32_t box_bytes;  // bytes one tensor copy lands (box_rows * lines * 128)
  float scale_log2;    // scale * log2(e)
  unsigned long long wait_limit_ns;  // bound of every pipeline wait
  long long stall_tile;  // tests of the bounded waits: flattened tile whose copies are withheld (-1: none)
};

struct Layout {
  uint32_t bar, meta, rows, misc, qring, stage, total;
};

// Shared-memory carve-up; identical on host (sizing) and device (addressing).
// Swizzled (tensor-core) stages start on a 1 KiB boundary of the shared
// window, for which `total` keeps 1 KiB of slack.
PA_HD Layout make_layout(int stages, int q_slots, uint32_t q_bytes, uint32_t stage_bytes,
                         bool swizzled) {
  Layout L;
  uint32_t o = 0;
  L.bar = o;
  o += 8u * (2u * stages + 2u * q_slots);
  o = (o + 15u) & ~15u;
  L.meta = o;
  o += 32u * stages;
  L.rows = o;  // per stage: pool row of each tile row holding a new token
  o += 4u * kTile * stages;
  L.misc = o;
  o += 4u * 80u;
  o = (o + 127u) & ~127u;
  L.qring = o;
  o += q_slots * ((q_bytes + 127u) & ~127u);
  o = (o + 127u) & ~127u;
  L.stage = o;
  o += stages * stage_bytes + (swizzled ? 1024u : 0u);
  L.total = o;
  return L;
}

__device__ __forceinline__ int clamp_context(const DecodeParams& p, int s, bool report_it) {
  int c = __ldg(p.context_lens + s);
  const int cmax = p.max_blocks_per_seq * p.block_size;
  if (c < 0 || c > cmax) {
    if (report_it) report(p.error_flag, PA_DEVERR_CONTEXT_LEN);
    c = c < 0 ? 0 : cmax;
  }
  return c;
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ long long warp_incl_scan_ll(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// ---------------------------------------------------------------------------
// Consumer state and tile math.  One consumer warp = one KV head and its G
// query heads; D = head size.
// ---------------------------------------------------------------------------

// Stages of the tensor-core consumers.  A K or V half-stage holds the tile's
// 16 token rows, row r as `lines` 128-byte lines (the head group's bytes,
// then zero-filled lines up to an odd count or the count a copy's alignment
// needs), written by tensor copies with the 128-byte swizzle: line
// L = r * lines + chunk stores its 16-byte unit u at position u ^ (L % 8).
// With `lines` odd, one unit of 8 consecutive rows lands in 8 different bank
// groups, so ldmatrix reads are conflict-free.
//
// RowPtr<NC> holds one lane's ldmatrix row address for a head whose bytes
// span NC 128-byte chunks: units u0 + 2j (j = 0, 1, ...) of row r, where u0
// counts 16-byte units from the start of the group's row and has bits 1-2
// clear, so stepping j within a chunk flips address bits 5-6 only.
template <int NC>
struct RowPtr {
  uint32_t a[NC];
  __device__ __forceinline__ RowPtr(uint32_t half, int r, int u0, uint32_t lines) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint32_t unit = (uint32_t)u0 + 8u * c;
      const uint32_t L = (uint32_t)r * lines + (unit >> 3);
      a[c] = half + L * kLine + (((unit & 7u) ^ (L & 7u)) << 4);
    }
  }
  __device__ __forceinline__ uint32_t at(int j) const { return a[j >> 2] ^ ((uint32_t)(j & 3) << 5); }
};

// bf16 tensor-core consumer.  Lane l owns query heads hA = 2*(l%4), hB = hA+1
// (columns of the score fragment) and, per 16-wide slice mt of the head
// dimension, output dims mt*16 + l/4 and +8.
template <int D>
struct MmaConsumer {
  static constexpr int KS = D / 16;  // k-steps of Q.K and m-tiles of P.V
  uint32_t qb[KS][2];
  float acc[KS][4];
  float m_a, m_b, l_a, l_b;

  __device__ __forceinline__ void begin_segment(const unsigned char* qslot, int w, int G,
                                                int lane) {
    const int n = lane >> 2, t2 = 2 * (lane & 3);
    const __nv_bfloat16* qh =
        reinterpret_cast<const __nv_bfloat16*>(qslot) + (size_t)(w * G + n) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (n < G) {
        qb[ks][0] = *reinterpret_cast<const uint32_t*>(qh + ks * 16 + t2);
        qb[ks][1] = *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 8 + t2);
      } else {
        qb[ks][0] = 0u;
        qb[ks][1] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[ks][i] = 0.f;
    }
    m_a = m_b = -INFINITY;
    l_a = l_b = 0.f;
  }

  static constexpr int NC = D * 2 > 128 ? D * 2 / 128 : 1;  // 128-byte chunks per head

  // k_half / v_half: the stage's K and V halves; uh: first 16-byte unit of
  // this warp's head within the group's row.
  __device__ __forceinline__ void tile(uint32_t k_half, uint32_t v_half, uint32_t lines, int uh,
                                       int nvalid, float scale_log2, int lane) {
    // S^T = K_tile * Q^T : rows = tokens, columns = query heads.
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const RowPtr<NC> kp(k_half, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(a, kp.at(ks));
      if (ks & 1)
        mma_bf16_16816(c1, a, qb[ks][0], qb[ks][1]);
      else
        mma_bf16_16816(c0, a, qb[ks][0], qb[ks][1]);
    }
    const int r0 = lane >> 2;
    float s0 = (c0[0] + c1[0]) * scale_log2, s1 = (c0[1] + c1[1]) * scale_log2;
    float s2 = (c0[2] + c1[2]) * scale_log2, s3 = (c0[3] + c1[3]) * scale_log2;
    if (r0 >= nvalid) s0 = s1 = -INFINITY;
    if (r0 + 8 >= nvalid) s2 = s3 = -INFINITY;

    // Online softmax: per-head tile maximum across the 8 lanes sharing l%4.
    float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    // A tile always holds a valid token, so mn_* is finite unless the inputs
    // are not; guard the exponent base anyway so -inf - -inf never appears.
    const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
    const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
    const float alpha_a = ex2_ftz(m_a - base_a), alpha_b = ex2_ftz(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    const float p0 = ex2_ftz(s0 - base_a), p1 = ex2_ftz(s1 - base_b);
    const float p2 = ex2_ftz(s2 - base_a), p3 = ex2_ftz(s3 - base_b);
    // P enters the bf16 MMA as a high and a low bf16 part (P = hi + lo to
    // about 2^-16), so the weights keep fp32-like precision.
    const uint32_t p_top = pack_bf16x2(p0, p1), p_bot = pack_bf16x2(p2, p3);
    const uint32_t r_top = pack_bf16x2(p0 - bf16_lo(p_top), p1 - bf16_hi(p_top));
    const uint32_t r_bot = pack_bf16x2(p2 - bf16_lo(p_bot), p3 - bf16_hi(p_bot));
    l_a = l_a * alpha_a + p0 + p2;
    l_b = l_b * alpha_b + p1 + p3;
    const uint32_t pb0 = movmatrix_trans(p_top);  // P^T rows (tokens) 0-7
    const uint32_t pb1 = movmatrix_trans(p_bot);  // tokens 8-15
    const uint32_t rb0 = movmatrix_trans(r_top);
    const uint32_t rb1 = movmatrix_trans(r_bot);

    // O^T += V^T * P^T : rows = head dims, columns = query heads.
    const RowPtr<NC> vp(v_half, (lane & 7) + (lane >> 4) * 8, uh + ((lane >> 3) & 1), lines);
    const int t2 = 2 * (lane & 3);
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (nvalid < kTile) {
      // Zero V entries of tokens past the end so stale stage contents (which
      // may be non-finite) never meet a zero weight.
      keep_lo = (t2 < nvalid ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid ? 0xffff0000u : 0u);
      keep_hi = (t2 + 8 < nvalid ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vp.at(mt));
      a[0] &= keep_lo;
      a[1] &= keep_lo;
      a[2] &= keep_hi;
      a[3] &= keep_hi;
      acc[mt][0] *= alpha_a;
      acc[mt][1] *= alpha_b;
      acc[mt][2] *= alpha_a;
      acc[mt][3] *= alpha_b;
      mma_bf16_16816(acc[mt], a, pb0, pb1);
      mma_bf16_16816(acc[mt], a, rb0, rb1);
    }
  }

  // slot < 0: final output; else partial slot of range r.
  __device__ __forceinline__ void finish(const DecodeParams& p, int seq, int kv_head, int slot,
                                         int r, int lane) {
    float la = l_a, lb = l_b;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, o);
      lb += __shfl_xor_sync(0xffffffffu, lb, o);
    }
    const int G = p.group, H = p.num_heads;
    const int ha = 2 * (lane & 3), hb = ha + 1, d0 = lane >> 2;
    const int qa = kv_head * G + ha, qb_ = kv_head * G + hb;
    if (slot < 0) {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)seq * H * D;
      const float ia = 1.f / la, ib = 1.f / lb;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d = mt * 16 + d0;
        if (ha < G) {
          out[(size_t)qa * D + d] = __float2bfloat16_rn(acc[mt][0] * ia);
          out[(size_t)qa * D + d + 8] = __float2bfloat16_rn(acc[mt][2] * ia);
        }
        if (hb < G) {
          out[(size_t)qb_ * D + d] = __float2bfloat16_rn(acc[mt][1] * ib);
          out[(size_t)qb_ * D + d + 8] = __float2bfloat16_rn(acc[mt][3] * ib);
        }
      }
    } else {
      const size_t base = ((size_t)r * 2 + slot) * H;
      float* po = p.part_o + base * D;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d = mt * 16 + d0;
        if (ha < G) {
          po[(size_t)qa * D + d] = acc[mt][0];
          po[(size_t)qa * D + d + 8] = acc[mt][2];
        }
        if (hb < G) {
          po[(size_t)qb_ * D + d] = acc[mt][1];
          po[(size_t)qb_ * D + d + 8] = acc[mt][3];
        }
      }
      if (d0 == 0) {
        float* pm = p.part_ml + base * 2;
        if (ha < G) {
          pm[(size_t)qa * 2 + 0] = m_a;
          pm[(size_t)qa * 2 + 1] = la;
        }
        if (hb < G) {
          pm[(size_t)qb_ * 2 + 0] = m_b;
          pm[(size_t)qb_ * 2 + 1] = lb;
        }
      }
    }
  }
};

// bf16 tensor-core consumer for several query tokens per sequence (causal).
// The N extent of the score fragment holds (query, head) columns: column
// n = qi * G + g for query qi < Q and group head g < G, NT tiles of 8 columns.
// Query qi sits at position ctx - Q + qi and sees tokens up to that position.
template <int D, int NT>
struct MmaConsumerMQ {
  static constexpr int KS = D / 16;
  uint32_t qb[NT][KS][2];
  float acc[NT][KS][4];
  float m_a[NT], m_b[NT], l_a[NT], l_b[NT];
  int col0 = 0;  // first (query, head) column this warp owns

  // w: KV head within the CTA's group; col_base: first column of this warp.
  __device__ __forceinline__ void begin_segment(const unsigned char* qslot, int w, int G, int Q,
                                                int Hg, int lane, int col_base) {
    col0 = col_base;
    const int t2 = 2 * (lane & 3);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = col0 + nt * 8 + (lane >> 2);
      const bool real = n < G * Q;
      const int qi = real ? n / G : 0, g = real ? n % G : 0;
      const __nv_bfloat16* qh =
          reinterpret_cast<const __nv_bfloat16*>(qslot) + ((size_t)qi * Hg * G + w * G + g) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[nt][ks][0] = real ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + t2) : 0u;
        qb[nt][ks][1] = real ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 8 + t2) : 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][ks][i] = 0.f;
      }
      m_a[nt] = m_b[nt] = -INFINITY;
      l_a[nt] = l_b[nt] = 0.f;
    }
  }

  // After a segment's finish (and merge) every state register is rewritten
  // by the next begin_segment before it is read; writing them here tells the
  // compiler so, which frees them for the merge.
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[nt][ks][0] = qb[nt][ks][1] = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][ks][i] = 0.f;
      }
      m_a[nt] = m_b[nt] = l_a[nt] = l_b[nt] = 0.f;
    }
  }

  static constexpr int NC = D * 2 > 128 ? D * 2 / 128 : 1;

  __device__ __forceinline__ void tile(uint32_t k_half, uint32_t v_half, uint32_t lines, int uh,
                                       int nvalid, int tok0, int ctx, int G, int Q,
                                       float scale_log2, int lane) {
    // Scores accumulate in two independent chains (even / odd k-steps) that
    // are added at the end: with one 8-column tile per warp, a single chain
    // would serialise all KS MMAs.
    float c[NT][4], c2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nt][i] = c2[nt][i] = 0.f;
    const RowPtr<NC> kp(k_half, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(a, kp.at(ks));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816((ks & 1) ? c2[nt] : c[nt], a, qb[nt][ks][0], qb[nt][ks][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[nt][i] += c2[nt][i];
    const int r0 = lane >> 2;
    const int t0 = tok0 + r0, t1 = t0 + 8;
    uint32_t pb0[NT], pb1[NT], rb0[NT], rb1[NT];
    float alpha_a[NT], alpha_b[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float s0 = c[nt][0] * scale_log2, s1 = c[nt][1] * scale_log2;
      float s2 = c[nt][2] * scale_log2, s3 = c[nt][3] * scale_log2;
      if (r0 >= nvalid) s0 = s1 = -INFINITY;
      if (r0 + 8 >= nvalid) s2 = s3 = -INFINITY;
      // Causal limits matter only on tiles that reach the queries' own
      // positions (ctx - Q ..); the test is the same for the whole warp.
      if (tok0 + kTile > ctx - Q) {
        const int na = col0 + nt * 8 + 2 * (lane & 3), nb = na + 1;
        // Last visible position of each column's query (-1: padding column).
        const int lim_a = na < G * Q ? ctx - Q + na / G : -1;
        const int lim_b = nb < G * Q ? ctx - Q + nb / G : -1;
        if (t0 > lim_a) s0 = -INFINITY;
        if (t0 > lim_b) s1 = -INFINITY;
        if (t1 > lim_a) s2 = -INFINITY;
        if (t1 > lim_b) s3 = -INFINITY;
      }
      float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
      }
      const float mn_a = fmaxf(m_a[nt], mx_a), mn_b = fmaxf(m_b[nt], mx_b);
      // A column may see no token of this tile (or none yet): keep -inf out of
      // the exponent base.
      const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
      const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
      alpha_a[nt] = ex2_ftz(m_a[nt] - base_a);
      alpha_b[nt] = ex2_ftz(m_b[nt] - base_b);
      m_a[nt] = mn_a;
      m_b[nt] = mn_b;
      const float p0 = ex2_ftz(s0 - base_a), p1 = ex2_ftz(s1 - base_b);
      const float p2 = ex2_ftz(s2 - base_a), p3 = ex2_ftz(s3 - base_b);
      const uint32_t p_top = pack_bf16x2(p0, p1), p_bot = pack_bf16x2(p2, p3);
      const uint32_t r_top = pack_bf16x2(p0 - bf16_lo(p_top), p1 - bf16_hi(p_top));
      const uint32_t r_bot = pack_bf16x2(p2 - bf16_lo(p_bot), p3 - bf16_hi(p_bot));
      l_a[nt] = l_a[nt] * alpha_a[nt] + p0 + p2;
      l_b[nt] = l_b[nt] * alpha_b[nt] + p1 + p3;
      pb0[nt] = movmatrix_trans(p_top);
      pb1[nt] = movmatrix_trans(p_bot);
      rb0[nt] = movmatrix_trans(r_top);
      rb1[nt] = movmatrix_trans(r_bot);
    }
    const RowPtr<NC> vp(v_half, (lane & 7) + (lane >> 4) * 8, uh + ((lane >> 3) & 1), lines);
    const int t2 = 2 * (lane & 3);
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (nvalid < kTile) {
      keep_lo = (t2 < nvalid ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid ? 0xffff0000u : 0u);
      keep_hi = (t2 + 8 < nvalid ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid ? 0xffff0000u : 0u);
    }
    // Rescale the accumulators only when some running max moved (a warp vote).
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) moved |= (alpha_a[nt] != 1.f) || (alpha_b[nt] != 1.f);
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[nt][mt][0] *= alpha_a[nt];
          acc[nt][mt][1] *= alpha_b[nt];
          acc[nt][mt][2] *= alpha_a[nt];
          acc[nt][mt][3] *= alpha_b[nt];
        }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vp.at(mt));
      a[0] &= keep_lo;
      a[1] &= keep_lo;
      a[2] &= keep_hi;
      a[3] &= keep_hi;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(acc[nt][mt], a, pb0[nt], pb1[nt]);
        mma_bf16_16816(acc[nt][mt], a, rb0[nt], rb1[nt]);
      }
    }
  }

  // The same with all K fragments loaded first, the scores in four chains
  // and the V fragments loaded before the softmax (used when a KV head's
  // columns are split over several warps, where it measured faster).
  __device__ __forceinline__ void tile_hoisted(uint32_t k_half, uint32_t v_half, uint32_t lines, int uh,
                                               int nvalid, int tok0, int ctx, int G, int Q,
                                       float scale_log2, int lane) {
    // All K fragments are loaded first, then the scores accumulate in four
    // independent chains (k-step mod 4) added at the end: with one 8-column
    // tile per warp a single chain would serialise all KS MMAs.  The V
    // fragments are loaded right after, so their latency overlaps the softmax.
    constexpr int NCH = KS < 4 ? KS : 4;
    uint32_t kf[KS][4], vf[KS][4];
    const RowPtr<NC> kp(k_half, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) ldmatrix_x4(kf[ks], kp.at(ks));
    float cc[NCH][NT][4];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) cc[ch][nt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(cc[ks % NCH][nt], kf[ks], qb[nt][ks][0], qb[nt][ks][1]);
    const RowPtr<NC> vp(v_half, (lane & 7) + (lane >> 4) * 8, uh + ((lane >> 3) & 1), lines);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) ldmatrix_x4_trans(vf[mt], vp.at(mt));
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = cc[0][nt][i];
#pragma unroll
        for (int ch = 1; ch < NCH; ++ch) v += cc[ch][nt][i];
        c[nt][i] = v;
      }
    const int r0 = lane >> 2;
    const int t0 = tok0 + r0, t1 = t0 + 8;
    uint32_t pb0[NT], pb1[NT], rb0[NT], rb1[NT];
    float alpha_a[NT], alpha_b[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float s0 = c[nt][0] * scale_log2, s1 = c[nt][1] * scale_log2;
      float s2 = c[nt][2] * scale_log2, s3 = c[nt][3] * scale_log2;
      if (r0 >= nvalid) s0 = s1 = -INFINITY;
      if (r0 + 8 >= nvalid) s2 = s3 = -INFINITY;
      // Causal limits matter only on tiles that reach the queries' own
      // positions (ctx - Q ..); the test is the same for the whole warp.
      if (tok0 + kTile > ctx - Q) {
        const int na = col0 + nt * 8 + 2 * (lane & 3), nb = na + 1;
        // Last visible position of each column's query (-1: padding column).
        const int lim_a = na < G * Q ? ctx - Q + na / G : -1;
        const int lim_b = nb < G * Q ? ctx - Q + nb / G : -1;
        if (t0 > lim_a) s0 = -INFINITY;
        if (t0 > lim_b) s1 = -INFINITY;
        if (t1 > lim_a) s2 = -INFINITY;
        if (t1 > lim_b) s3 = -INFINITY;
      }
      float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
      }
      const float mn_a = fmaxf(m_a[nt], mx_a), mn_b = fmaxf(m_b[nt], mx_b);
      // A column may see no token of this tile (or none yet): keep -inf out of
      // the exponent base.
      const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
      const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
      alpha_a[nt] = ex2_ftz(m_a[nt] - base_a);
      alpha_b[nt] = ex2_ftz(m_b[nt] - base_b);
      m_a[nt] = mn_a;
      m_b[nt] = mn_b;
      const float p0 = ex2_ftz(s0 - base_a), p1 = ex2_ftz(s1 - base_b);
      const float p2 = ex2_ftz(s2 - base_a), p3 = ex2_ftz(s3 - base_b);
      const uint32_t p_top = pack_bf16x2(p0, p1), p_bot = pack_bf16x2(p2, p3);
      const uint32_t r_top = pack_bf16x2(p0 - bf16_lo(p_top), p1 - bf16_hi(p_top));
      const uint32_t r_bot = pack_bf16x2(p2 - bf16_lo(p_bot), p3 - bf16_hi(p_bot));
      l_a[nt] = l_a[nt] * alpha_a[nt] + p0 + p2;
      l_b[nt] = l_b[nt] * alpha_b[nt] + p1 + p3;
      pb0[nt] = movmatrix_trans(p_top);
      pb1[nt] = movmatrix_trans(p_bot);
      rb0[nt] = movmatrix_trans(r_top);
      rb1[nt] = movmatrix_trans(r_bot);
    }
    const int t2 = 2 * (lane & 3);
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (nvalid < kTile) {
      keep_lo = (t2 < nvalid ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid ? 0xffff0000u : 0u);
      keep_hi = (t2 + 8 < nvalid ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid ? 0xffff0000u : 0u);
    }
    // Rescale the accumulators only when some running max moved (a warp vote).
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) moved |= (alpha_a[nt] != 1.f) || (alpha_b[nt] != 1.f);
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[nt][mt][0] *= alpha_a[nt];
          acc[nt][mt][1] *= alpha_b[nt];
          acc[nt][mt][2] *= alpha_a[nt];
          acc[nt][mt][3] *= alpha_b[nt];
        }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      vf[mt][0] &= keep_lo;
      vf[mt][1] &= keep_lo;
      vf[mt][2] &= keep_hi;
      vf[mt][3] &= keep_hi;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt][mt], vf[mt], pb0[nt], pb1[nt]);
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt][mt], vf[mt], rb0[nt], rb1[nt]);
  }

  // Two consecutive tiles of one segment in one pass (the first full, from
  // tok0; the second with nvalid1 tokens from tok0 + 16): the two tiles'
  // score chains interleave and one softmax update covers all 32 tokens.
  __device__ __forceinline__ void tile2(uint32_t k_half0, uint32_t v_half0, uint32_t k_half1, uint32_t v_half1,
                                        uint32_t lines, int uh, int nvalid1, int tok0, int ctx, int G, int Q,
                                        float scale_log2, int lane) {
    const RowPtr<NC> kp0(k_half0, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines);
    const RowPtr<NC> kp1(k_half1, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines);
    float cc[2][2][NT][4];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) cc[tt][ch][nt][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a0[4], a1[4];
      ldmatrix_x4(a0, kp0.at(ks));
      ldmatrix_x4(a1, kp1.at(ks));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(cc[0][ks & 1][nt], a0, qb[nt][ks][0], qb[nt][ks][1]);
        mma_bf16_16816(cc[1][ks & 1][nt], a1, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }
    const int r0 = lane >> 2;
    uint32_t pb[2][NT][4];  // per tile: P^T hi rows 0-7, 8-15, then lo rows 0-7, 8-15
    float alpha_a[NT], alpha_b[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sv[2][4];
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int nv = tt ? nvalid1 : kTile;
#pragma unroll
        for (int i = 0; i < 4; ++i) sv[tt][i] = (cc[tt][0][nt][i] + cc[tt][1][nt][i]) * scale_log2;
        if (r0 >= nv) sv[tt][0] = sv[tt][1] = -INFINITY;
        if (r0 + 8 >= nv) sv[tt][2] = sv[tt][3] = -INFINITY;
      }
      if (tok0 + 2 * kTile > ctx - Q) {  // the pair reaches the queries' own positions
        const int na = col0 + nt * 8 + 2 * (lane & 3), nb = na + 1;
        const int lim_a = na < G * Q ? ctx - Q + na / G : -1;
        const int lim_b = nb < G * Q ? ctx - Q + nb / G : -1;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          const int t0 = tok0 + 16 * tt + r0, t1 = t0 + 8;
          if (t0 > lim_a) sv[tt][0] = -INFINITY;
          if (t0 > lim_b) sv[tt][1] = -INFINITY;
          if (t1 > lim_a) sv[tt][2] = -INFINITY;
          if (t1 > lim_b) sv[tt][3] = -INFINITY;
        }
      }
      float mx_a = fmaxf(fmaxf(sv[0][0], sv[0][2]), fmaxf(sv[1][0], sv[1][2]));
      float mx_b = fmaxf(fmaxf(sv[0][1], sv[0][3]), fmaxf(sv[1][1], sv[1][3]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
      }
      const float mn_a = fmaxf(m_a[nt], mx_a), mn_b = fmaxf(m_b[nt], mx_b);
      const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
      const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
      alpha_a[nt] = ex2_ftz(m_a[nt] - base_a);
      alpha_b[nt] = ex2_ftz(m_b[nt] - base_b);
      m_a[nt] = mn_a;
      m_b[nt] = mn_b;
      float la = 0.f, lb = 0.f;
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const float p0 = ex2_ftz(sv[tt][0] - base_a), p1 = ex2_ftz(sv[tt][1] - base_b);
        const float p2 = ex2_ftz(sv[tt][2] - base_a), p3 = ex2_ftz(sv[tt][3] - base_b);
        const uint32_t p_top = pack_bf16x2(p0, p1), p_bot = pack_bf16x2(p2, p3);
        const uint32_t r_top = pack_bf16x2(p0 - bf16_lo(p_top), p1 - bf16_hi(p_top));
        const uint32_t r_bot = pack_bf16x2(p2 - bf16_lo(p_bot), p3 - bf16_hi(p_bot));
        la += p0 + p2;
        lb += p1 + p3;
        pb[tt][nt][0] = movmatrix_trans(p_top);
        pb[tt][nt][1] = movmatrix_trans(p_bot);
        pb[tt][nt][2] = movmatrix_trans(r_top);
        pb[tt][nt][3] = movmatrix_trans(r_bot);
      }
      l_a[nt] = l_a[nt] * alpha_a[nt] + la;
      l_b[nt] = l_b[nt] * alpha_b[nt] + lb;
    }
    const int t2 = 2 * (lane & 3);
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (nvalid1 < kTile) {
      keep_lo = (t2 < nvalid1 ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid1 ? 0xffff0000u : 0u);
      keep_hi = (t2 + 8 < nvalid1 ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid1 ? 0xffff0000u : 0u);
    }
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) moved |= (alpha_a[nt] != 1.f) || (alpha_b[nt] != 1.f);
    if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[nt][mt][0] *= alpha_a[nt];
          acc[nt][mt][1] *= alpha_b[nt];
          acc[nt][mt][2] *= alpha_a[nt];
          acc[nt][mt][3] *= alpha_b[nt];
        }
    }
    const RowPtr<NC> vp0(v_half0, (lane & 7) + (lane >> 4) * 8, uh + ((lane >> 3) & 1), lines);
    const RowPtr<NC> vp1(v_half1, (lane & 7) + (lane >> 4) * 8, uh + ((lane >> 3) & 1), lines);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t v0[4], v1[4];
      ldmatrix_x4_trans(v0, vp0.at(mt));
      ldmatrix_x4_trans(v1, vp1.at(mt));
      v1[0] &= keep_lo;
      v1[1] &= keep_lo;
      v1[2] &= keep_hi;
      v1[3] &= keep_hi;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(acc[nt][mt], v0, pb[0][nt][0], pb[0][nt][1]);
        mma_bf16_16816(acc[nt][mt], v1, pb[1][nt][0], pb[1][nt][1]);
        mma_bf16_16816(acc[nt][mt], v0, pb[0][nt][2], pb[0][nt][3]);
        mma_bf16_16816(acc[nt][mt], v1, pb[1][nt][2], pb[1][nt][3]);
      }
    }
  }

  // Output rows are [seq][query][head]; partial rows are [query][head].
  __device__ __forceinline__ void finish(const DecodeParams& p, int seq, int kv_head, int slot,
                                         int r, int lane) {
    const int G = p.group, H = p.num_heads, Q = p.num_queries;
    const int d0 = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float la = l_a[nt], lb = l_b[nt];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, o);
        lb += __shfl_xor_sync(0xffffffffu, lb, o);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int n = col0 + nt * 8 + 2 * (lane & 3) + half;
        if (n >= G * Q) continue;
        const int qi = n / G, g = n % G;
        const int row = qi * H + kv_head * G + g;
        const float l = half ? lb : la, m = half ? m_b[nt] : m_a[nt];
        if (slot < 0) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)seq * Q * H + row) * D;
          const float inv = l > 0.f ? 1.f / l : 0.f;  // a query with no keys gives zeros
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            out[mt * 16 + d0] = __float2bfloat16_rn(acc[nt][mt][half] * inv);
            out[mt * 16 + d0 + 8] = __float2bfloat16_rn(acc[nt][mt][2 + half] * inv);
          }
        } else {
          const size_t base = ((size_t)r * 2 + slot) * Q * H + row;
          float* po = p.part_o + base * D;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            po[mt * 16 + d0] = acc[nt][mt][half];
            po[mt * 16 + d0 + 8] = acc[nt][mt][2 + half];
          }
          if (d0 == 0) {
            p.part_ml[base * 2 + 0] = m;
            p.part_ml[base * 2 + 1] = l;
          }
        }
      }
    }
  }
};

// Consumer for an FP8 (E4M3) pool with bf16 queries and outputs.  Codes are
// widened to f16 in registers (exact) and both products run on f16 MMAs.
// Shared-memory reads use ldmatrix on 16-bit units (two codes each):
//   Q.K  - the order of head dims inside each 16-wide k-step is permuted so
//          that lane t's four consecutive codes (dims 4t..4t+3) are its k
//          pairs (2t, 2t+1) and (2t+8, 2t+9); the query fragment is loaded in
//          the same order, so the sum is unchanged.
//   P.V  - ldmatrix.trans hands each lane two dims of two tokens; the MMA's
//          output rows are permuted so that lane l/4 owns dims 2*(l/4) and
//          +1 of each 16-wide slice, and one byte permute per register builds
//          the (token, token) pairs the A operand needs.
// Scores carry k_scale in scale_log2; v_scale is applied to the output.  The
// bf16 query converts to f16 exactly for |q| in f16's normal range
// [2^-14, 65504]; P enters as f16.
// MQ: several query tokens per sequence with a causal mask, as in
// MmaConsumerMQ: column n = col0 + (lane / 4) holds (query n / G, head n % G),
// query qi sits at position ctx - Q + qi and sees tokens up to it.
template <int D, bool MQ = false>
struct MmaConsumerF8 {
  static constexpr int KS = D / 16;
  uint32_t qb[KS][2];
  float acc[KS][4];
  float m_a, m_b, l_a, l_b;
  uint32_t lane_off = 0;  // this lane's ldmatrix row address within a half-stage (K and V alike)
  int col0 = 0;           // MQ: first (query, head) column of this warp

  // Once per kernel: uh is the head's first 16-byte unit in the group's row.
  __device__ __forceinline__ void setup(uint32_t lines, int uh, int lane) {
    lane_off = RowPtr<1>(0u, (lane & 7) + ((lane >> 3) & 1) * 8, uh + (lane >> 4), lines).a[0];
  }

  // w: KV head within the CTA's group.  MQ also takes Q, Hg and this warp's
  // first column.
  __device__ __forceinline__ void begin_segment(const unsigned char* qslot, int w, int G, int lane,
                                                int Q = 1, int Hg = 1, int col_base = 0) {
    const int t4 = 4 * (lane & 3);
    const __nv_bfloat16* qh;
    bool real;
    if constexpr (MQ) {
      col0 = col_base;
      const int n = col_base + (lane >> 2);
      real = n < G * Q;
      const int qi = real ? n / G : 0, g = real ? n % G : 0;
      qh = reinterpret_cast<const __nv_bfloat16*>(qslot) + ((size_t)qi * Hg * G + w * G + g) * D;
    } else {
      const int n = lane >> 2;
      real = n < G;
      qh = reinterpret_cast<const __nv_bfloat16*>(qslot) + (size_t)(w * G + n) * D;
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (real) {
        const uint2 v = *reinterpret_cast<const uint2*>(qh + ks * 16 + t4);  // dims t4 .. t4+3
        qb[ks][0] = pack_f16x2(bf16_lo(v.x), bf16_hi(v.x));  // k pair (2t, 2t+1)
        qb[ks][1] = pack_f16x2(bf16_lo(v.y), bf16_hi(v.y));  // k pair (2t+8, 2t+9)
      } else {
        qb[ks][0] = 0u;
        qb[ks][1] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[ks][i] = 0.f;
    }
    m_a = m_b = -INFINITY;
    l_a = l_b = 0.f;
  }

  // After a segment's finish (and merge) every state register is rewritten
  // by the next begin_segment before it is read; writing them here tells the
  // compiler so, which frees them for the merge.
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = qb[ks][1] = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[ks][i] = 0.f;
    }
    m_a = m_b = l_a = l_b = 0.f;
  }

  // MQ: tok0 (first token of the tile), ctx, G and Q give the causal limits.
  __device__ __forceinline__ void tile(uint32_t k_half, uint32_t v_half, int nvalid, float scale_log2,
                                       int lane, int tok0 = 0, int ctx = 0, int G = 1, int Q = 1) {
    // Matrices of one ldmatrix.x4: (rows 0-7, bytes 0-15), (rows 8-15, 0-15),
    // (rows 0-7, 16-31), (rows 8-15, 16-31) - two k-steps / m-tiles of 16 dims.
    // Half-stages are 1 KiB aligned, so adding the lane offset keeps the
    // swizzled unit bits that at(j)'s XOR steps through.
    const uint32_t ka = k_half + lane_off, va = v_half + lane_off;
    uint32_t kr[KS / 2][4], vr[KS / 2][4];
#pragma unroll
    for (int j = 0; j < KS / 2; ++j) ldmatrix_x4(kr[j], ka ^ ((uint32_t)(j & 3) << 5));
#pragma unroll
    for (int j = 0; j < KS / 2; ++j) ldmatrix_x4_trans(vr[j], va ^ ((uint32_t)(j & 3) << 5));

    // Scores accumulate in four independent chains (k-step mod 4).
    constexpr int NCH = KS < 4 ? KS : 4;
    float cc[NCH][4];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
      for (int i = 0; i < 4; ++i) cc[ch][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint32_t top = kr[ks >> 1][2 * (ks & 1)], bot = kr[ks >> 1][2 * (ks & 1) + 1];
      uint32_t a[4];
      e4m3x4_to_f16x2x2(top, a[0], a[2]);  // token row g: codes 0,1 | codes 2,3
      e4m3x4_to_f16x2x2(bot, a[1], a[3]);  // token row g+8
      mma_f16_16816(cc[ks % NCH], a, qb[ks][0], qb[ks][1]);
    }
#pragma unroll
    for (int ch = 1; ch < NCH; ++ch)
#pragma unroll
      for (int i = 0; i < 4; ++i) cc[0][i] += cc[ch][i];
    const int g = lane >> 2, t2 = 2 * (lane & 3);
    float s0 = cc[0][0] * scale_log2, s1 = cc[0][1] * scale_log2;
    float s2 = cc[0][2] * scale_log2, s3 = cc[0][3] * scale_log2;
    if (g >= nvalid) s0 = s1 = -INFINITY;
    if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
    if (MQ && tok0 + kTile > ctx - Q) {  // only tiles reaching the queries' own positions
      // Last visible position of each column's query (-1: padding column).
      const int na = col0 + t2, nb = na + 1;
      const int lim_a = na < G * Q ? ctx - Q + na / G : -1;
      const int lim_b = nb < G * Q ? ctx - Q + nb / G : -1;
      const int t0 = tok0 + g, t1 = t0 + 8;
      if (t0 > lim_a) s0 = -INFINITY;
      if (t0 > lim_b) s1 = -INFINITY;
      if (t1 > lim_a) s2 = -INFINITY;
      if (t1 > lim_b) s3 = -INFINITY;
    }
    float mx_a = fmaxf(s0, s2), mx_b = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
    const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
    const float alpha_a = ex2_ftz(m_a - base_a), alpha_b = ex2_ftz(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    const float p0 = ex2_ftz(s0 - base_a), p1 = ex2_ftz(s1 - base_b);
    const float p2 = ex2_ftz(s2 - base_a), p3 = ex2_ftz(s3 - base_b);
    // Weights enter the f16 MMA rounded to f16 (relative error <= 2^-11,
    // half an ulp of the 10-bit fraction), well inside the bf16 output's own
    // rounding; the running sum keeps them in fp32.
    const uint32_t p_top = pack_f16x2(p0, p1), p_bot = pack_f16x2(p2, p3);
    l_a = l_a * alpha_a + p0 + p2;
    l_b = l_b * alpha_b + p1 + p3;
    const uint32_t pb0 = movmatrix_trans(p_top), pb1 = movmatrix_trans(p_bot);
    // Each V register holds bytes (tok 2t: dim 2g, 2g+1 | tok 2t+1: dim 2g, 2g+1);
    // on the last tile of a segment, tokens past the end are zeroed (code 0
    // is +0.0) before they meet a weight.
    if (nvalid < kTile) {
      const uint32_t keep_lo = (t2 < nvalid ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid ? 0xffff0000u : 0u);
      const uint32_t keep_hi = (t2 + 8 < nvalid ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
      for (int j = 0; j < KS / 2; ++j) {
        vr[j][0] &= keep_lo;
        vr[j][1] &= keep_hi;
        vr[j][2] &= keep_lo;
        vr[j][3] &= keep_hi;
      }
    }
    // Once the running maxima settle, most tiles leave every alpha at 1:
    // skip the rescale then (this consumer is issue-bound).
    if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[mt][0] *= alpha_a;
        acc[mt][1] *= alpha_b;
        acc[mt][2] *= alpha_a;
        acc[mt][3] *= alpha_b;
      }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const uint32_t top = vr[mt >> 1][2 * (mt & 1)];      // tokens 2t, 2t+1
      const uint32_t bot = vr[mt >> 1][2 * (mt & 1) + 1];  // tokens 2t+8, 2t+9
      // One byte permute per register: (dim 2g: tokens 2t, 2t+1 | dim 2g+1: same).
      uint32_t a[4];
      e4m3x4_to_f16x2x2(__byte_perm(top, 0u, 0x3120), a[0], a[1]);
      e4m3x4_to_f16x2x2(__byte_perm(bot, 0u, 0x3120), a[2], a[3]);
      mma_f16_16816(acc[mt], a, pb0, pb1);
    }
  }

  // Two consecutive tiles of one segment in one pass: the first full (16
  // tokens from tok0), the second holding nvalid1 tokens from tok0 + 16.  Their
  // score MMAs interleave in four independent chains and one softmax update
  // covers all 32 tokens, so the fixed-latency steps (score reductions,
  // exponentials, rescale) run once per pair.
  __device__ __forceinline__ void tile2(uint32_t k_half0, uint32_t v_half0, uint32_t k_half1, uint32_t v_half1,
                                        int nvalid1, float scale_log2, int lane, int tok0 = 0, int ctx = 0,
                                        int G = 1, int Q = 1) {
    const uint32_t ka[2] = {k_half0 + lane_off, k_half1 + lane_off};
    const uint32_t va[2] = {v_half0 + lane_off, v_half1 + lane_off};
    uint32_t kr[2][KS / 2][4];
#pragma unroll
    for (int j = 0; j < KS / 2; ++j)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) ldmatrix_x4(kr[tt][j], ka[tt] ^ ((uint32_t)(j & 3) << 5));
    float cc[2][2][4];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int i = 0; i < 4; ++i) cc[tt][ch][i] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const uint32_t top = kr[tt][ks >> 1][2 * (ks & 1)], bot = kr[tt][ks >> 1][2 * (ks & 1) + 1];
        uint32_t a[4];
        e4m3x4_to_f16x2x2(top, a[0], a[2]);
        e4m3x4_to_f16x2x2(bot, a[1], a[3]);
        mma_f16_16816(cc[tt][ks & 1], a, qb[ks][0], qb[ks][1]);
      }
    uint32_t vr[2][KS / 2][4];
#pragma unroll
    for (int j = 0; j < KS / 2; ++j)
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) ldmatrix_x4_trans(vr[tt][j], va[tt] ^ ((uint32_t)(j & 3) << 5));
    const int g = lane >> 2, t2 = 2 * (lane & 3);
    float sc[2][4];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[tt][i] = (cc[tt][0][i] + cc[tt][1][i]) * scale_log2;
    if (g >= nvalid1) sc[1][0] = sc[1][1] = -INFINITY;
    if (g + 8 >= nvalid1) sc[1][2] = sc[1][3] = -INFINITY;
    if (MQ && tok0 + 2 * kTile > ctx - Q) {  // the pair reaches the queries' own positions
      const int na = col0 + t2, nb = na + 1;
      const int lim_a = na < G * Q ? ctx - Q + na / G : -1;
      const int lim_b = nb < G * Q ? ctx - Q + nb / G : -1;
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int t0 = tok0 + 16 * tt + g, t1 = t0 + 8;
        if (t0 > lim_a) sc[tt][0] = -INFINITY;
        if (t0 > lim_b) sc[tt][1] = -INFINITY;
        if (t1 > lim_a) sc[tt][2] = -INFINITY;
        if (t1 > lim_b) sc[tt][3] = -INFINITY;
      }
    }
    float mx_a = fmaxf(fmaxf(sc[0][0], sc[0][2]), fmaxf(sc[1][0], sc[1][2]));
    float mx_b = fmaxf(fmaxf(sc[0][1], sc[0][3]), fmaxf(sc[1][1], sc[1][3]));
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, o));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, o));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float base_a = (mn_a == -INFINITY) ? 0.f : mn_a;
    const float base_b = (mn_b == -INFINITY) ? 0.f : mn_b;
    const float alpha_a = ex2_ftz(m_a - base_a), alpha_b = ex2_ftz(m_b - base_b);
    m_a = mn_a;
    m_b = mn_b;
    float pw[2][4];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      pw[tt][0] = ex2_ftz(sc[tt][0] - base_a);
      pw[tt][1] = ex2_ftz(sc[tt][1] - base_b);
      pw[tt][2] = ex2_ftz(sc[tt][2] - base_a);
      pw[tt][3] = ex2_ftz(sc[tt][3] - base_b);
    }
    l_a = l_a * alpha_a + ((pw[0][0] + pw[0][2]) + (pw[1][0] + pw[1][2]));
    l_b = l_b * alpha_b + ((pw[0][1] + pw[0][3]) + (pw[1][1] + pw[1][3]));
    uint32_t pb[2][2];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
      pb[tt][0] = movmatrix_trans(pack_f16x2(pw[tt][0], pw[tt][1]));
      pb[tt][1] = movmatrix_trans(pack_f16x2(pw[tt][2], pw[tt][3]));
    }
    if (nvalid1 < kTile) {
      const uint32_t keep_lo = (t2 < nvalid1 ? 0x0000ffffu : 0u) | (t2 + 1 < nvalid1 ? 0xffff0000u : 0u);
      const uint32_t keep_hi = (t2 + 8 < nvalid1 ? 0x0000ffffu : 0u) | (t2 + 9 < nvalid1 ? 0xffff0000u : 0u);
#pragma unroll
      for (int j = 0; j < KS / 2; ++j) {
        vr[1][j][0] &= keep_lo;
        vr[1][j][1] &= keep_hi;
        vr[1][j][2] &= keep_lo;
        vr[1][j][3] &= keep_hi;
      }
    }
    if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[mt][0] *= alpha_a;
        acc[mt][1] *= alpha_b;
        acc[mt][2] *= alpha_a;
        acc[mt][3] *= alpha_b;
      }
    }
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const uint32_t top = vr[tt][mt >> 1][2 * (mt & 1)];
        const uint32_t bot = vr[tt][mt >> 1][2 * (mt & 1) + 1];
        uint32_t a[4];
        e4m3x4_to_f16x2x2(__byte_perm(top, 0u, 0x3120), a[0], a[1]);
        e4m3x4_to_f16x2x2(__byte_perm(bot, 0u, 0x3120), a[2], a[3]);
        mma_f16_16816(acc[mt], a, pb[tt][0], pb[tt][1]);
      }
  }

  // Output row pairs: acc[mt][0] / [2] are dims dd / dd+1 of column a,
  // [1] / [3] of column b.  Output rows are [seq][query][head]; partial rows
  // are [query][head] (one query: [head]).
  __device__ __forceinline__ void finish(const DecodeParams& p, int seq, int kv_head, int slot,
                                         int r, int lane) {
    float la = l_a, lb = l_b;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, o);
      lb += __shfl_xor_sync(0xffffffffu, lb, o);
    }
    const int G = p.group, H = p.num_heads, Q = MQ ? p.num_queries : 1;
    const int g = lane >> 2;
    if constexpr (!MQ) {
      const int ha = 2 * (lane & 3), hb = ha + 1;
      const int qa = kv_head * G + ha, qb_ = kv_head * G + hb;
      if (slot < 0) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)seq * H * D;
        const float ia = p.v_scale / la, ib = p.v_scale / lb;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int dd = mt * 16 + 2 * g;
          if (ha < G)
            *reinterpret_cast<uint32_t*>(out + (size_t)qa * D + dd) = pack_bf16x2(acc[mt][0] * ia, acc[mt][2] * ia);
          if (hb < G)
            *reinterpret_cast<uint32_t*>(out + (size_t)qb_ * D + dd) = pack_bf16x2(acc[mt][1] * ib, acc[mt][3] * ib);
        }
      } else {
        const size_t base = ((size_t)r * 2 + slot) * H;
        float* po = p.part_o + base * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int dd = mt * 16 + 2 * g;
          if (ha < G) *reinterpret_cast<float2*>(po + (size_t)qa * D + dd) = make_float2(acc[mt][0], acc[mt][2]);
          if (hb < G) *reinterpret_cast<float2*>(po + (size_t)qb_ * D + dd) = make_float2(acc[mt][1], acc[mt][3]);
        }
        if (g == 0) {
          float* pm = p.part_ml + base * 2;
          if (ha < G) *reinterpret_cast<float2*>(pm + (size_t)qa * 2) = make_float2(m_a, la);
          if (hb < G) *reinterpret_cast<float2*>(pm + (size_t)qb_ * 2) = make_float2(m_b, lb);
        }
      }
    } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int n = col0 + 2 * (lane & 3) + half;
        if (n >= G * Q) continue;
        int qi = 0, gh = n;
        if constexpr (MQ) {
          qi = n / G;
          gh = n % G;
        }
        const int row = qi * H + kv_head * G + gh;
        const float l = half ? lb : la, m = half ? m_b : m_a;
        if (slot < 0) {
          __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)seq * Q * H + row) * D;
          // A query with no keys (several queries, short context) gives zeros.
          const float inv = (!MQ || l > 0.f) ? p.v_scale / l : 0.f;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
            *reinterpret_cast<uint32_t*>(out + mt * 16 + 2 * g) =
                pack_bf16x2(acc[mt][half] * inv, acc[mt][2 + half] * inv);
        } else {
          const size_t base = ((size_t)r * 2 + slot) * Q * H + row;
          float* po = p.part_o + base * D;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
            *reinterpret_cast<float2*>(po + mt * 16 + 2 * g) = make_float2(acc[mt][half], acc[mt][2 + half]);
          if (g == 0) *reinterpret_cast<float2*>(p.part_ml + base * 2) = make_float2(m, l);
        }
      }
    }
  }
};

// fp32 CUDA-core consumer.  Lane l owns head dims [l*DC, l*DC+DC) of every
// query head; after the butterfly reduction lane l holds the score of token l/2.
template <int D, int GMAX>
struct SimtConsumer {
  static constexpr int DC = D / 32;
  float qv[GMAX][DC];
  float acc[GMAX][DC];
  float m[GMAX], l[GMAX];  // l: this lane's share (token l/2, counted on even and odd lanes)

  __device__ __forceinline__ void begin_segment(const unsigned char* qslot, int w, int G,
                                                int lane) {
    const float* qh = reinterpret_cast<const float*>(qslot) + (size_t)w * G * D;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
#pragma unroll
      for (int i = 0; i < DC; ++i) {
        qv[h][i] = (h < G) ? qh[(size_t)h * D + lane * DC + i] : 0.f;
        acc[h][i] = 0.f;
      }
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
  }

  __device__ __forceinline__ void tile(const unsigned char* k_base, const unsigned char* v_base,
                                       uint32_t pitch, int nvalid, float scale_log2, int G,
                                       int lane) {
    const int my_tok = lane >> 1;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h >= G) break;
      float part[kTile];
#pragma unroll
      for (int t = 0; t < kTile; ++t) {
        const float* kr = reinterpret_cast<const float*>(k_base + t * pitch) + lane * DC;
        float sacc = 0.f;
#pragma unroll
        for (int i = 0; i < DC; ++i) sacc = fmaf(qv[h][i], kr[i], sacc);
        part[t] = sacc;
      }
      // Butterfly reduce-scatter: 16 partial sums over 32 lanes -> one full sum
      // per lane pair.  Step xor 16 keeps the half selected by lane bit 4, etc.
      float v8[8], v4[4], v2[2];
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float mine = b4 ? part[i + 8] : part[i];
        const float give = b4 ? part[i] : part[i + 8];
        v8[i] = mine + __shfl_xor_sync(0xffffffffu, give, 16);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float mine = b3 ? v8[i + 4] : v8[i];
        const float give = b3 ? v8[i] : v8[i + 4];
        v4[i] = mine + __shfl_xor_sync(0xffffffffu, give, 8);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float mine = b2 ? v4[i + 2] : v4[i];
        const float give = b2 ? v4[i] : v4[i + 2];
        v2[i] = mine + __shfl_xor_sync(0xffffffffu, give, 4);
      }
      float sc;
      {
        const float mine = b1 ? v2[1] : v2[0];
        const float give = b1 ? v2[0] : v2[1];
        sc = mine + __shfl_xor_sync(0xffffffffu, give, 2);
      }
      sc += __shfl_xor_sync(0xffffffffu, sc, 1);
      sc *= scale_log2;
      if (my_tok >= nvalid) sc = -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m[h], mx);
      const float base = (mn == -INFINITY) ? 0.f : mn;
      const float alpha = ex2_ftz(m[h] - base);
      m[h] = mn;
      const float pw = ex2_ftz(sc - base);
      l[h] = l[h] * alpha + pw;
#pragma unroll
      for (int i = 0; i < DC; ++i) acc[h][i] *= alpha;
      for (int t = 0; t < nvalid; ++t) {
        const float pt = __shfl_sync(0xffffffffu, pw, 2 * t);
        const float* vr = reinterpret_cast<const float*>(v_base + t * pitch) + lane * DC;
#pragma unroll
        for (int i = 0; i < DC; ++i) acc[h][i] = fmaf(pt, vr[i], acc[h][i]);
      }
    }
  }

  __device__ __forceinline__ void finish(const DecodeParams& p, int seq, int kv_head, int slot,
                                         int r, int lane) {
    const int G = p.group, H = p.num_heads;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      if (h >= G) break;
      float lt = l[h];
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, o);
      const int qh = kv_head * G + h;
      if (slot < 0) {
        float* out = reinterpret_cast<float*>(p.out) + ((size_t)seq * H + qh) * D + lane * DC;
        const float inv = 1.f / lt;
#pragma unroll
        for (int i = 0; i < DC; ++i) out[i] = acc[h][i] * inv;
      } else {
        const size_t base = ((size_t)r * 2 + slot) * H + qh;
        float* po = p.part_o + base * D + lane * DC;
#pragma unroll
        for (int i = 0; i < DC; ++i) po[i] = acc[h][i];
        if (lane == 0) {
          p.part_ml[base * 2 + 0] = m[h];
          p.part_ml[base * 2 + 1] = lt;
        }
      }
    }
  }
};

// Zero the output rows of an empty sequence (16-byte stores; rows are 16-byte multiples).
template <typename T, int D>
__device__ void zero_row(const DecodeParams& p, int s) {
  // Output rows of sequence s: [num_queries][num_heads][D].
  const size_t n = (size_t)p.num_queries * p.num_heads * D;
  const size_t n16 = n * sizeof(T) / 16;
  uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) + (size_t)s * n);
  for (size_t i = 0; i < n16; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Called by a consumer warp right after it wrote its partial (m, l, O) for
// (seq, kv_head).  Takes a ticket; the warp holding the last of the r1-r0+1
// tickets merges every partial of that sequence and KV head by log-sum-exp,
// writes the output rows, and resets the ticket counter.  Nobody waits.
// `arrivals`: warps writing partials per range and KV head (two to four when
// the (query, head) columns of a KV head are split across several warps).
template <typename T, int D, bool kMQ>
__device__ void arrive_and_merge(const DecodeParams& p, int seq, int kv_head, int r0, int r1,
                                 int slot0, int lane, int arrivals = 1) {
  // Release: the warp barrier orders every lane's partial stores before lane
  // 0's fence, which makes them visible device-wide before the ticket.
  // Acquire: the warp holding the last ticket fences before the barrier that
  // releases its lanes to read the other partials.
  const int last = arrivals * (r1 - r0 + 1) - 1;
  int* cnt = p.counters + (size_t)seq * p.num_kv_heads + kv_head;
  __syncwarp();
  int ticket = 0;
  if (lane == 0) {
    __threadfence();
    ticket = atomicAdd(cnt, 1);
    if (ticket == last) __threadfence();
  }
  __syncwarp();
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  if (ticket != last) return;
  // Online pass over the partials, four query heads of this KV head at a
  // time: lane l owns dims [l*DL, l*DL+DL) of each head.  The next partial's
  // loads are issued before the current one is folded in.
  constexpr int DL = D / 32;
  constexpr int GM = 4;
  const int G = p.group, H = kMQ ? p.num_queries * p.num_heads : p.num_heads;
  const int nq = kMQ ? p.num_queries : 1;
  for (int gq = 0, gn = 0; gq < G * nq; gq += gn) {
    // Rows of this KV head, at most four at a time and never across queries:
    // query qi, group heads g0 .. g0 + gn - 1.
    const int qi = gq / G, g0 = gq % G;
    const int h0 = qi * p.num_heads + kv_head * G + g0;
    gn = min(GM, G - g0);
    float run_m[GM], run_l[GM], acc[GM][DL];
    float nm[GM], nl[GM], no[GM][DL];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      run_m[g] = -INFINITY;
      run_l[g] = 0.f;
#pragma unroll
      for (int i = 0; i < DL; ++i) acc[g][i] = 0.f;
    }
    auto load = [&](int rr) {
      const int sl = rr == r0 ? slot0 : 0;
      const size_t base = ((size_t)rr * 2 + sl) * H + h0;
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < gn) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + base + g);
          nm[g] = ml.x;
          nl[g] = ml.y;
          const float* po = p.part_o + (base + g) * D + lane * DL;
          if constexpr (DL == 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(po));
            no[g][0] = v.x; no[g][1] = v.y; no[g][2] = v.z; no[g][3] = v.w;
          } else {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(po));
            no[g][0] = v.x; no[g][1] = v.y;
          }
        }
      }
    };
    load(r0);
    for (int rr = r0; rr <= r1; ++rr) {
      float cm[GM], cl[GM], co[GM][DL];
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        cm[g] = nm[g];
        cl[g] = nl[g];
#pragma unroll
        for (int i = 0; i < DL; ++i) co[g][i] = no[g][i];
      }
      if (rr < r1) load(rr + 1);
#pragma unroll
      for (int g = 0; g < GM; ++g) {
        if (g < gn) {
          const float mnew = fmaxf(run_m[g], cm[g]);
          // Several queries: a query may have no keys in some (or all)
          // partials, m = -inf; keep -inf out of the exponent base.
          const float mb = (kMQ && mnew == -INFINITY) ? 0.f : mnew;
          const float a_old = ex2_ftz(run_m[g] - mb), a_new = ex2_ftz(cm[g] - mb);
          run_m[g] = mnew;
          run_l[g] = run_l[g] * a_old + cl[g] * a_new;
#pragma unroll
          for (int i = 0; i < DL; ++i) acc[g][i] = acc[g][i] * a_old + co[g][i] * a_new;
        }
      }
    }
    T* out = reinterpret_cast<T*>(p.out) + ((size_t)seq * H + h0) * D + lane * DL;
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < gn) {
        const float inv = (kMQ && run_l[g] == 0.f) ? 0.f : p.v_scale / run_l[g];
#pragma unroll
        for (int i = 0; i < DL; ++i) out[(size_t)g * D + i] = T(acc[g][i] * inv);
      }
    }
  }
  __syncwarp();
  if (lane == 0) *cnt = 0;  // leave the counter zeroed for the next call
}

// Appending calls: a tile holding some of the step's new tokens (tile rows
// mt.newfirst .. mt.nvalid - 1, query positions c - Q .. c - 1) may have been
// staged before those tokens reached the pool, so the warp of KV head kv_head
// puts each new token's K and V (from k_new / v_new, row s * Q + i for the
// token at position c - Q + i) into its own columns of the staged rows,
// swizzled as the tensor copy lays them out, and also stores them into the
// token's pool row (rows[r]; -1 leaves it unwritten).  Lane u < 16 moves
// 16-byte unit u of the K row, lane 16 + u the same unit of V.
template <int D>
__device__ __forceinline__ void append_new_rows(const DecodeParams& p, const StageMeta& mt, const int* rows,
                                                int kv_head, int w, uint32_t k_half, uint32_t v_half,
                                                int lane) {
  constexpr int UH = D * 2 / 16;  // 16-byte units of one head's bf16 row
  const int u = lane & 15;
  const bool is_v = lane >= 16;
  const int Q = p.num_queries;
  for (int r = mt.newfirst; r < mt.nvalid; ++r) {
    const int prow = rows[r];
    if (u < UH && prow >= 0) {
      const size_t tok = (size_t)mt.seq * Q + (mt.tok0 + r - (mt.ctx - Q));  // row of k_new / v_new
      const size_t e = (tok * p.num_kv_heads + kv_head) * D + u * 8;
      const uint4 val = __ldg(reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(is_v ? p.v_new : p.k_new) + e));
      const uint32_t unit = (uint32_t)(w * UH + u);
      const uint32_t L = (uint32_t)r * p.lines + (unit >> 3);
      const uint32_t dst = (is_v ? v_half : k_half) + L * kLine + (((unit & 7u) ^ (L & 7u)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(val.x), "r"(val.y),
                   "r"(val.z), "r"(val.w)
                   : "memory");
      __nv_bfloat16* pool = static_cast<__nv_bfloat16*>(const_cast<void*>(is_v ? p.v_cache : p.k_cache));
      *reinterpret_cast<uint4*>(pool + ((size_t)prow * p.num_kv_heads + kv_head) * D + u * 8) = val;
    }
  }
  // The stage is later refilled by the TMA engine (async proxy): order these
  // generic-proxy writes before that, and make them visible to the warp.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// The same for FP8 pools (one query per sequence): the token's bf16 K/V are
// quantised exactly as the FP8 cache write does (fp32 quotient by the pool's
// scale, E4M3 round to nearest even, saturating), 16 codes per lane.
template <int D>
__device__ __forceinline__ void append_new_rows_fp8(const DecodeParams& p, const StageMeta& mt,
                                                    const int* rows, int kv_head, int w, uint32_t k_half,
                                                    uint32_t v_half, int lane) {
  constexpr int UH = D / 16;  // 16-byte units of one head's FP8 row
  const int u = lane & 15;
  const bool is_v = lane >= 16;
  const int Q = p.num_queries;
  for (int r = mt.newfirst; r < mt.nvalid; ++r) {
    const int prow = rows[r];
    if (u < UH && prow >= 0) {
      const size_t tok = (size_t)mt.seq * Q + (mt.tok0 + r - (mt.ctx - Q));
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(is_v ? p.v_new : p.k_new) + (tok * p.num_kv_heads + kv_head) * D +
          u * 16);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      const float sc = is_v ? p.v_scale : p.k_scale;
      const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
            make_float2(bf16_lo(in[2 * i]) / sc, bf16_hi(in[2 * i]) / sc), __NV_SATFINITE, __NV_E4M3));
        const uint32_t hi = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
            make_float2(bf16_lo(in[2 * i + 1]) / sc, bf16_hi(in[2 * i + 1]) / sc), __NV_SATFINITE, __NV_E4M3));
        out[i] = lo | (hi << 16);
      }
      const uint32_t unit = (uint32_t)(w * UH + u);
      const uint32_t L = (uint32_t)r * p.lines + (unit >> 3);
      const uint32_t dst = (is_v ? v_half : k_half) + L * kLine + (((unit & 7u) ^ (L & 7u)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(out[0]), "r"(out[1]),
                   "r"(out[2]), "r"(out[3])
                   : "memory");
      unsigned char* pool = static_cast<unsigned char*>(const_cast<void*>(is_v ? p.v_cache : p.k_cache));
      *reinterpret_cast<uint4*>(pool + ((size_t)prow * p.num_kv_heads + kv_head) * D + u * 16) =
          make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Kernel 1
// ---------------------------------------------------------------------------
// QMODE 0: one query per sequence.  QMODE 1 / 2: several query tokens per
// sequence with a causal mask, (query, head) columns in one 8-wide MMA N-tile
// per warp: one warp per KV head (up to 8 columns) or p.split warps (2 to 4,
// up to 32 columns).
template <typename T, int D, int GMAX, int QMODE, bool KV8 = false>
__global__ void __launch_bounds__(32 * (kMaxGroupHeads + kProducers), 1)
    pa_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int HG = p.num_head_groups, R = p.num_ranges, S = p.num_seqs;
  const int r = blockIdx.x / HG, hg = blockIdx.x % HG;
  const int Hg = p.heads_per_cta;
  // QMODE 2 splits each KV head's (query, head) columns over p.split warps,
  // 8 columns each (up to 32 columns: four warps).
  const int kSplit = QMODE == 2 ? p.split : 1;
  const int NCW = Hg * kSplit;  // consumer warps; warps NCW .. NCW + kProducers - 1 produce
  constexpr bool kMmaPath = (sizeof(T) == 2);  // tensor-core consumers, swizzled stages
  const Layout L = make_layout(p.stages, p.q_slots, p.q_bytes, p.stage_bytes, kMmaPath);
  long long* misc = reinterpret_cast<long long*>(smem + L.misc);  // [0,32) scratch, [32..] results
  griddep_wait();  // inputs may come from the kernel just before (e.g. the cache write)

  // ---- Prologue: total tile count, this range, and its first sequence. ----
  long long total = 0;
  for (int base = 0; base < S; base += nthreads) {
    const int s = base + tid;
    long long n = (s < S) ? tiles_of(clamp_context(p, s, true)) : 0;
    if (s < S && n == 0 && s % gridDim.x == blockIdx.x) zero_row<T, D>(p, s);
    n = warp_sum_ll(n);
    if (lane == 0) misc[warp] = n;
    __syncthreads();
    for (int w = 0; w < nwarps; ++w) total += misc[w];
    __syncthreads();
  }
  // Never more ranges than tiles, so no range is empty and a cut sequence
  // has exactly r1 - r0 + 1 partials.
  const long long Reff = total < R ? total : R;
  if (r >= Reff) return;
  const long long a = range_start(r, total, Reff), b = range_start(r + 1, total, Reff);

  long long run = 0;
  for (int base = 0; base < S; base += nthreads) {
    const int s = base + tid;
    const long long n = (s < S) ? tiles_of(clamp_context(p, s, false)) : 0;
    const long long incl = warp_incl_scan_ll(n, lane);
    if (lane == 31) misc[warp] = incl;
    __syncthreads();
    long long before = run;
    for (int w = 0; w < warp; ++w) before += misc[w];
    long long chunk = 0;
    for (int w = 0; w < nwarps; ++w) chunk += misc[w];
    const long long excl = before + incl - n;
    if (s < S && n > 0 && excl <= a && a < excl + n) {
      misc[32] = s;
      misc[33] = excl;
    }
    run += chunk;
    __syncthreads();
  }
  griddep_launch_dependents();  // the next kernel may get resident; it waits for our completion

  const uint32_t bar0 = smem_addr(smem + L.bar);
  const int NS = p.stages, NQ = p.q_slots;
  auto full_bar = [&](int i) { return bar0 + 8u * i; };
  auto empty_bar = [&](int i) { return bar0 + 8u * (NS + i); };
  auto qfull_bar = [&](int i) { return bar0 + 8u * (2 * NS + i); };
  auto qempty_bar = [&](int i) { return bar0 + 8u * (2 * NS + NQ + i); };
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta);
  int* stage_rows = reinterpret_cast<int*>(smem + L.rows);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 34);
  // A pipeline wait ran out: report it and tell the producers to drain.
  auto timed_out = [&]() {
    if (lane == 0) {
      report(p.error_flag, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  };
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), NCW);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(qfull_bar(i), 1);
      mbar_init(qempty_bar(i), NCW);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  const int s_first = static_cast<int>(misc[32]);
  const long long p_first = misc[33];
  const uint32_t q_slot_bytes = (p.q_bytes + 127u) & ~127u;
  const uint32_t qring = smem_addr(smem + L.qring);
  const uint32_t stages =
      kMmaPath ? ((smem_addr(smem + L.stage) + 1023u) & ~1023u) : smem_addr(smem + L.stage);
  const int G = p.group, H = p.num_heads, Hk = p.num_kv_heads, bs = p.block_size;

  if (warp >= NCW) {
    // ---------------- producers ----------------
    const int pw = warp - NCW;  // this producer takes the tiles x with (x - a) % kProducers == pw
    // Pool element: T, or one byte for an FP8 pool.
    using KV = typename std::conditional<KV8, unsigned char, T>::type;
    const KV* kc = reinterpret_cast<const KV*>(p.k_cache);
    const KV* vc = reinterpret_cast<const KV*>(p.v_cache);
    const T* qg = reinterpret_cast<const T*>(p.q);
    int s = s_first;
    long long ps = p_first;
    int c = clamp_context(p, s, false);
    long long ns = tiles_of(c);
    // The next sequence's length is fetched one sequence ahead.
    int c_next = (s + 1 < S) ? clamp_context(p, s + 1, false) : 0;
    int slot = 0, seg_r0 = 0, seg_r1 = 0, seg_slot0 = 0;
    int st = 0, qi = 0;
    uint32_t ph = 0, qph = 0;
    // Stages and query slots this warp armed, with the parity of the last
    // phase it armed on each (for the drain after a timeout).
    uint32_t my_stages = 0u, my_stage_par = 0u, my_qs = 0u, my_q_par = 0u;
    const int t = lane & 15;
    const bool is_v = lane >= 16;
    if (kMmaPath && lane == 0) {
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
    }
    // Per-lane constants of the copy issue: whether this lane leads a copy
    // (tensor paths: the first row of a box), where in a stage its copy
    // lands, and which pool it reads.  Power-of-two block sizes take shifts
    // and masks instead of integer division.
    const bool lead = kMmaPath ? (t % (int)p.box_rows) == 0 : true;
    const uint32_t lane_dst = kMmaPath ? (is_v ? kTile * p.lines * kLine : 0u) + t * p.lines * kLine
                                       : (is_v ? kTile * p.pitch : 0u) + t * p.pitch;
    const void* tmap = is_v ? static_cast<const void*>(&p.tm_v) : static_cast<const void*>(&p.tm_k);
    const int bs_sh = (bs & (bs - 1)) == 0 ? __ffs(bs) - 1 : -1;
    auto blk_of = [&](int tok) { return bs_sh >= 0 ? tok >> bs_sh : tok / bs; };
    auto off_of = [&](int tok) { return bs_sh >= 0 ? tok & (bs - 1) : tok % bs; };
    // Block-table window of the current sequence: lane i holds entry cb+i in
    // `cur` and cb+32+i in `nxt`.  The window slides one chunk at a time and the
    // next chunk is loaded a chunk ahead, so lookups never wait on memory except
    // at the first tile of a segment.
    const int32_t* bt_row = nullptr;
    int nblk = 0, cb = 0, cur = -1, nxt = -1;
    auto table_entry = [&](int idx) -> int { return idx < nblk ? __ldg(bt_row + idx) : -1; };
    for (long long x = a; x < b; ++x) {
      bool new_seq = (x == a);
      while (x >= ps + ns) {
        ps += ns;
        ++s;
        c = c_next;
        ns = tiles_of(c);
        c_next = (s + 1 < S) ? clamp_context(p, s + 1, false) : 0;
        new_seq = true;
      }
      const int j = static_cast<int>(x - ps);
      const int tok0 = j * kTile;
      const int nvalid = min(kTile, c - tok0);
      const int blk0 = blk_of(tok0);
      if (new_seq) {
        slot = segment_slot(a, b, ps, ps + ns);
        if (slot >= 0) {
          seg_r0 = static_cast<int>(range_of_tile(ps, total, Reff));
          seg_r1 = static_cast<int>(range_of_tile(ps + ns - 1, total, Reff));
          seg_slot0 = partial_slot_of_range(seg_r0, ps, total, Reff);
        }
        bt_row = p.block_tables + (size_t)s * p.max_blocks_per_seq;
        nblk = (c + bs - 1) / bs;
        cb = blk0;
        cur = table_entry(cb + lane);
        nxt = table_entry(cb + 32 + lane);
      }
      while (blk0 >= cb + 32) {
        cur = nxt;
        cb += 32;
        nxt = table_entry(cb + 32 + lane);
      }
      const int flags = (new_seq ? kSegBegin : 0) | ((x == b - 1 || j == ns - 1) ? kSegEnd : 0) |
                        ((slot + 1) << 2) | (seg_slot0 << 4);
      const bool mine = kProducers == 1 || static_cast<int>((x - a) % kProducers) == pw;
      if (new_seq && mine) {
        if (!mbar_wait_warp(qempty_bar(qi), qph ^ 1u, p.wait_limit_ns)) {
          timed_out();
          break;
        }
        if (lane == 0) {
          const uint32_t qb = qfull_bar(qi);
          mbar_arrive_expect_tx(qb, p.q_bytes);
          if constexpr (QMODE == 0) {
            bulk_copy_g2s(qring + qi * q_slot_bytes, qg + ((size_t)s * H + (size_t)hg * Hg * G) * D,
                          p.q_bytes, qb);
          } else {
            // Query rows are [seq][query][head]: one copy per query token.
            const uint32_t per_q = p.q_bytes / p.num_queries;
            for (int qq = 0; qq < p.num_queries; ++qq)
              bulk_copy_g2s(qring + qi * q_slot_bytes + qq * per_q,
                            qg + (((size_t)s * p.num_queries + qq) * H + (size_t)hg * Hg * G) * D,
                            per_q, qb);
          }
        }
        my_qs |= 1u << qi;
        my_q_par = (my_q_par & ~(1u << qi)) | (qph << qi);
      }
      if (new_seq && ++qi == NQ) {  // every producer follows the query ring
        qi = 0;
        qph ^= 1u;
      }
      if (!mine) {  // the other producer's tile: only follow the stage ring
        if (++st == NS) {
          st = 0;
          ph ^= 1u;
        }
        continue;
      }
      // This lane's token -> physical block (a tile spans at most 16 blocks, so
      // it always lies inside the 64-entry window).
      const int tok = tok0 + t;
      const int rel = blk_of(tok) - cb;
      const int e_cur = __shfl_sync(0xffffffffu, cur, rel & 31);
      const int e_nxt = __shfl_sync(0xffffffffu, nxt, rel & 31);
      const int phys = rel < 32 ? e_cur : e_nxt;
      bool ok = t < nvalid;
      if (ok && p.num_physical_blocks > 0 && (phys < 0 || phys >= p.num_physical_blocks)) {
        report(p.error_flag, PA_DEVERR_BLOCK_ID);
        ok = false;
      }
      // Tensor-core paths: lane t (t a multiple of box_rows) copies tile rows
      // t .. t + box_rows - 1, which lie in one block, as one tensor box; rows
      // past the context in that block come along and are masked by the
      // consumers.  fp32: one bulk copy per valid token row.
      ok = ok && lead;
      const unsigned copies = __ballot_sync(0xffffffffu, ok);
      // Token row of the pool: fewer than 2^31 in any pool that fits in device memory.
      const int row = (int)((bs_sh >= 0 ? (unsigned)phys << bs_sh : (unsigned)phys * (unsigned)bs) +
                            (unsigned)off_of(tok));
      // Appending calls: the step's new tokens are positions c - Q .. c - 1.
      int newfirst = -1;
      if (kMmaPath && p.k_new != nullptr && tok0 + nvalid > c - p.num_queries) {
        newfirst = max(0, c - p.num_queries - tok0);
      }
      if (!mbar_wait_warp(empty_bar(st), ph ^ 1u, p.wait_limit_ns)) {
        timed_out();
        break;
      }
      // Tests of the bounded waits: this tile's stage is never armed or
      // filled, so the consumers' wait on it runs out.
      const bool stall = x == p.stall_tile;
      if (newfirst >= 0 && !is_v && t >= newfirst && t < nvalid) {
        // Pool row of this tile row's new token; a failed block check leaves it unwritten.
        const bool bad = p.num_physical_blocks > 0 && (phys < 0 || phys >= p.num_physical_blocks);
        stage_rows[st * kTile + t] = bad ? -1 : row;
      }
      __syncwarp();
      if (lane == 0 && !stall) {
        meta[st] = StageMeta{s, tok0, nvalid, flags, seg_r0, seg_r1, c, newfirst};
        mbar_arrive_expect_tx(full_bar(st), __popc(copies) * (kMmaPath ? p.box_bytes : p.row_bytes));
      }
      __syncwarp();
      if (!stall) {
        my_stages |= 1u << st;
        my_stage_par = (my_stage_par & ~(1u << st)) | (ph << st);
      }
      if (ok && !stall) {
        const uint32_t dst = stages + st * p.stage_bytes + lane_dst;
        if constexpr (kMmaPath) {
          tma_load_4d(dst, tmap, 0, 0, hg, row, full_bar(st));
        } else {
          const KV* src = (is_v ? vc : kc) + ((size_t)row * Hk + (size_t)hg * Hg) * D;
          bulk_copy_g2s(dst, src, p.row_bytes, full_bar(st));
        }
      }
      if (++st == NS) {
        st = 0;
        ph ^= 1u;
      }
    }
    named_barrier_sync(1, nthreads);  // every warp has left its tile loop
    if (*abort_flag != 0 && lane == 0) {
      // A wait ran out, so the loops ended early and copies this warp started
      // may still be landing.  Wait (again bounded) for the last phase it
      // armed on each stage and query slot, so that no copy writes into this
      // CTA's shared memory after it has retired.
      for (int i = 0; i < NS; ++i)
        if ((my_stages >> i) & 1u) (void)mbar_wait(full_bar(i), (my_stage_par >> i) & 1u, p.wait_limit_ns);
      for (int i = 0; i < NQ; ++i)
        if ((my_qs >> i) & 1u) (void)mbar_wait(qfull_bar(i), (my_q_par >> i) & 1u, p.wait_limit_ns);
    }
  } else {
    // ---------------- consumers ----------------
    const int w = warp / kSplit;  // KV head within the group
    const int col_base = (warp % kSplit) * 8;
    const int kv_head = hg * Hg + w;
    int st = 0, qi = 0;
    uint32_t ph = 0, qph = 0;
    constexpr bool kMma = (sizeof(T) == 2);
    using Mma = typename std::conditional<
        KV8, MmaConsumerF8<D, (QMODE > 0)>,
        typename std::conditional<QMODE == 0, MmaConsumer<D>, MmaConsumerMQ<D, 1>>::type>::type;
    typename std::conditional<kMma, Mma, SimtConsumer<D, GMAX>>::type cons;
    if constexpr (KV8) cons.setup(p.lines, w * D / 16, lane);
    // FP8 consumers, and bf16 ones that split a KV head's columns over
    // several warps, take two stages at a time when both hold the same
    // segment (tile pairing: tile2), if the ring has four or more stages.
    // Their tile math, not HBM, sets the pace.  One-query bf16 decode and
    // bf16 multi-query with one warp per KV head (2 KiB rows, a 3-stage ring
    // for the common shapes) are HBM-bound and keep the ring for copies.
    constexpr bool kPair = kMma && (KV8 || QMODE == 2);
    for (long long x = a; x < b; ++x) {
      if (!mbar_wait_warp(full_bar(st), ph, p.wait_limit_ns)) {
        timed_out();
        break;
      }
      const StageMeta mt = meta[st];
      if (mt.flags & kSegBegin) {
        if (!mbar_wait_warp(qfull_bar(qi), qph, p.wait_limit_ns)) {
          timed_out();
          break;
        }
        if constexpr (QMODE == 0)
          cons.begin_segment(smem + L.qring + qi * q_slot_bytes, w, G, lane);
        else if constexpr (KV8)
          cons.begin_segment(smem + L.qring + qi * q_slot_bytes, w, G, lane, p.num_queries, Hg, col_base);
        else
          cons.begin_segment(smem + L.qring + qi * q_slot_bytes, w, G, p.num_queries, Hg, lane,
                             col_base);
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty_bar(qi));
        if (++qi == NQ) {
          qi = 0;
          qph ^= 1u;
        }
      }
      constexpr int kKVBytes = KV8 ? 1 : (int)sizeof(T);
      const uint32_t k_half = stages + st * p.stage_bytes;
      const uint32_t v_half = k_half + kTile * p.lines * kLine;
      const int uh = w * D * kKVBytes / 16;  // this head's first 16-byte unit in the row
      if constexpr (kMma && QMODE < 2) {
        if (mt.newfirst >= 0) {
          const int* rows = stage_rows + st * kTile;
          if constexpr (KV8)
            append_new_rows_fp8<D>(p, mt, rows, kv_head, w, k_half, v_half, lane);
          else
            append_new_rows<D>(p, mt, rows, kv_head, w, k_half, v_half, lane);
        }
      }
      // A tile that does not end its segment is followed, in the next stage,
      // by the same segment's next tile: pair them.
      bool paired = false;
      StageMeta me = mt;  // the pass's last tile (it carries the segment end)
      int st_last = st;
      if constexpr (kPair) {
        // The ring has four or more stages here (the host plan checks it): a
        // pair holds two, and the copies need the rest.
        if (!(mt.flags & kSegEnd)) {
          const int st2 = st + 1 == NS ? 0 : st + 1;
          const uint32_t ph2 = st + 1 == NS ? ph ^ 1u : ph;
          if (!mbar_wait_warp(full_bar(st2), ph2, p.wait_limit_ns)) {
            timed_out();
            break;
          }
          me = meta[st2];
          const uint32_t k_half2 = stages + st2 * p.stage_bytes;
          const uint32_t v_half2 = k_half2 + kTile * p.lines * kLine;
          if constexpr (QMODE < 2) {
            if (me.newfirst >= 0) {
              if constexpr (KV8)
                append_new_rows_fp8<D>(p, me, stage_rows + st2 * kTile, kv_head, w, k_half2, v_half2, lane);
              else
                append_new_rows<D>(p, me, stage_rows + st2 * kTile, kv_head, w, k_half2, v_half2, lane);
            }
          }
          if constexpr (KV8 && QMODE > 0)
            cons.tile2(k_half, v_half, k_half2, v_half2, me.nvalid, p.scale_log2, lane, mt.tok0, mt.ctx, G,
                       p.num_queries);
          else if constexpr (KV8)
            cons.tile2(k_half, v_half, k_half2, v_half2, me.nvalid, p.scale_log2, lane);
          else
            cons.tile2(k_half, v_half, k_half2, v_half2, p.lines, uh, me.nvalid, mt.tok0, mt.ctx, G,
                       p.num_queries, p.scale_log2, lane);
          paired = true;
          st_last = st2;
          ++x;
        }
      }
      if (paired) {
      } else if constexpr (KV8 && QMODE > 0) {
        cons.tile(k_half, v_half, mt.nvalid, p.scale_log2, lane, mt.tok0, mt.ctx, G, p.num_queries);
      } else if constexpr (KV8) {
        cons.tile(k_half, v_half, mt.nvalid, p.scale_log2, lane);
      } else if constexpr (kMma && QMODE == 2) {
        cons.tile_hoisted(k_half, v_half, p.lines, uh, mt.nvalid, mt.tok0, mt.ctx, G, p.num_queries,
                          p.scale_log2, lane);
      } else if constexpr (kMma && QMODE > 0) {
        cons.tile(k_half, v_half, p.lines, uh, mt.nvalid, mt.tok0, mt.ctx, G, p.num_queries,
                  p.scale_log2, lane);
      } else if constexpr (kMma) {
        cons.tile(k_half, v_half, p.lines, uh, mt.nvalid, p.scale_log2, lane);
      } else {
        const unsigned char* kb = smem + L.stage + st * p.stage_bytes + w * D * sizeof(T);
        cons.tile(kb, kb + kTile * p.pitch, p.pitch, mt.nvalid, p.scale_log2, G, lane);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(empty_bar(st));
        if (paired) mbar_arrive(empty_bar(st_last));
      }
      if (me.flags & kSegEnd) {
        const int slot = ((me.flags >> 2) & 3) - 1;
        cons.finish(p, me.seq, kv_head, slot, r, lane);
        if (slot >= 0)
          arrive_and_merge<T, D, (QMODE > 0)>(p, me.seq, kv_head, me.r0, me.r1, (me.flags >> 4) & 1, lane,
                                              kSplit);
        // Split-column kernels sit at the register cap: writing the state here
        // (the next segment's begin_segment rewrites it anyway) frees its
        // registers for the merge above.
        if constexpr (QMODE == 2) cons.clear();
      }
      if (++st == NS) {
        st = 0;
        ph ^= 1u;
      }
      if (paired && ++st == NS) {
        st = 0;
        ph ^= 1u;
      }
    }
    named_barrier_sync(1, nthreads);  // lets the producers drain their copies after a timeout
  }
  (void)Hk;
}

}  // namespace pa
