// tcgen05 GEMM of the fused LM-head variant: one persistent kernel template serves the four
// contractions of the step ("Sizing mini-batches and micro-batches", "The problem": the logits
// of 2048-token completions over the whole vocabulary must never be held at once).
//
//   pass A      z = h W^T tile by tile, epilogue: per-row (shift, sum-exp) over the tile and the
//               target logit (EPI_PARTIALS)
//   recompute   the same product over one vocabulary chunk, epilogue: bf16 dlogits of the chunk
//               into a bounded chunk buffer (EPI_DLOGITS)
//   d_h         d_h (+)= dz_c W_c   A = dz_c K-major, B = W_c MN-major (EPI_STORE_F32)
//   dW          dW_c = dz_c^T h     A = dz_c MN-major, B = h MN-major  (EPI_STORE_F32)
//
// CG = 2 (the product instance): a 2-CTA cluster computes one 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M = 256). Each CTA loads its own 128 rows of A and its own 128 rows
// of B with plain TMA tile loads from this GPU's memory; the paired MMA reads both halves of B
// from the two CTAs' shared memory, so each CTA stages 32 KB per 64-wide K step instead of the
// 48 KB a one-CTA 128 x 256 tile needs. Each CTA's TMEM holds its 128 accumulator rows.
// CG = 1: the same tile shape per CTA without a cluster (one CTA computes 128 x 256).
//
// Warps: 0 = TMA producer (one thread), 1 = MMA issuer (one thread; with CG = 2 only the
// cluster's even CTA issues), 2..5 = epilogue (thread = TMEM lane = accumulator row). The
// shared-memory ring is STAGES deep; the TMEM accumulator is double-buffered (2 x 256 columns),
// so a tile's epilogue runs while the next tile's MMAs proceed. Every wait is bounded: a wait
// that gives up raises a flag, the kernel runs to its end and reports kFlagWaitTimeout.
#pragma once

#include <cuda.h>

#include "grpo_common.cuh"

namespace grpo {
namespace lmhead {

constexpr int BM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;  // accumulator columns per tile
constexpr int BK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int NTHREADS = 192;
constexpr int TMEM_COLS = 2 * BN;

// EPI_PARTIALS_ENT: the partials plus sum e z per tile (the entropy's third accumulator)
enum Epi : int { EPI_PARTIALS = 0, EPI_DLOGITS = 1, EPI_STORE_F32 = 2, EPI_PARTIALS_ENT = 3 };

// Dlogits epilogue staging: each epilogue warp writes its 32 rows x 32 columns of bf16 (2 KB,
// 64-byte rows in the 64-byte swizzle a TMA store expects) into one of two buffers, and one lane
// stores the box with a TMA tile store (full 64-byte row segments instead of 32 scattered
// 16-byte pieces per store instruction).
constexpr int EPI_BOX = 32;                          // rows and columns of a staged box
constexpr int EPI_BUF_BYTES = EPI_BOX * EPI_BOX * 2;  // 2 KB
constexpr int EPI_WARPS = 4;

template <int CG, int EPI = EPI_PARTIALS>
struct Shape {
  static constexpr int A_BYTES = BM * BK * 2;            // 16 KB
  static constexpr int B_ROWS = BN / CG;                 // rows of B this CTA stages
  static constexpr int B_BYTES = B_ROWS * BK * 2;        // 16 KB (CG = 2) or 32 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // bytes this CTA receives per stage
  static constexpr int STAGES = CG == 2 ? 6 : 4;
  static constexpr int EPI_BYTES = EPI == EPI_DLOGITS ? EPI_WARPS * 2 * EPI_BUF_BYTES : 0;
  static constexpr size_t SMEM = 1024 /*alignment slack*/ + (size_t)STAGES * STAGE_BYTES + EPI_BYTES + 256;
};

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16, the major-ness of each
// operand (0 = K-major, 1 = MN-major), N = 256, M = 128 * CG.
template <int CG, bool A_MN, bool B_MN>
constexpr uint32_t idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)A_MN << 15) | ((uint32_t)B_MN << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((BM * CG) >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzle (version 1). Operands are staged in
// 128-byte rows, 8-row swizzle atoms of 1024 bytes:
//  K-major  (rows = M or N, 64 K values per row): atoms along MN 1024 bytes apart (stride byte
//           offset); the leading byte offset is unused.
//  MN-major (rows = K, 64 MN values per row, one TMA box of 64 K rows per 64 MN columns):
//           8-row K groups 1024 bytes apart (stride byte offset), 64-wide MN blocks one box
//           (8192 bytes) apart (leading byte offset).
template <bool MN>
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((MN ? 8192u : 16u) >> 4) << 16;  // leading byte offset
  d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset
  d |= (uint64_t)1 << 46;                          // descriptor version
  d |= (uint64_t)2 << 61;                          // SWIZZLE_128B
  return d;
}

// Descriptor advance per 16-wide K step, in 16-byte units: 32 bytes along a K-major row, two
// 8-row K groups (2048 bytes) for MN-major.
template <bool MN>
constexpr uint64_t kstep() {
  return MN ? 128u : 2u;
}

// 2-D TMA tile load into this CTA's shared memory. `bar` is a shared::cluster address: this
// CTA's barrier, or with CG = 2 the barrier of the cluster's even CTA (which counts the bytes of
// both CTAs' loads).
template <int CG>
__device__ __forceinline__ void tma2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  if constexpr (CG == 1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
  }
}

// One operand tile of R rows (M or N) x 64 K values. K-major: one box {64 K, R rows} at
// (k0, mn0). MN-major: R / 64 boxes {64 MN, 64 K}, box i at (mn0 + 64 i, k0), 8192 bytes apart.
template <int CG, bool MN, int R>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar, int k0, int mn0) {
  if constexpr (MN) {
#pragma unroll
    for (int i = 0; i < R / 64; ++i) tma2d<CG>(dst + (uint32_t)i * 8192u, map, bar, mn0 + 64 * i, k0);
  } else {
    tma2d<CG>(dst, map, bar, k0, mn0);
  }
}

// 2-D TMA tile store from this CTA's shared memory (bulk-group completion); the parts of the
// box outside the tensor map's extents are not written.
__device__ __forceinline__ void tma_store2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most N of this thread's committed bulk groups may still be reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// this thread's generic-proxy shared-memory writes become visible to the async proxy (TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, bool accum) {
  if constexpr (CG == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"((uint32_t)accum)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"((uint32_t)accum)
        : "memory");
}

// Arrive on the mbarrier at shared::cluster address `bar` once every tcgen05.mma this thread
// issued so far has completed.
template <int CG>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot) {
  if constexpr (CG == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t tmem) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

// Bounded wait that ignores the abort flag: the end-of-kernel drain after a timeout.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) return;
  }
}

__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  __syncwarp();  // the load is warp-collective: reconverge lanes that skipped a store
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct GemmArgs {
  int64_t M, N, K;  // output rows and columns, reduction length
  int n_m, n_n;     // work units along M (BM * CG rows each) and N (BN columns each)
  int m_fast;       // unit order: 1 = consecutive units walk M (share the B tile), 0 = walk N
  int col_tile0;    // EPI_PARTIALS / EPI_DLOGITS: vocabulary tile of the launch's first column
  // EPI_PARTIALS / EPI_DLOGITS: rows are tokens (M = T), columns vocabulary entries (< V)
  int64_t V;
  const int32_t* target;
  float* part_m;  // [n_col_tiles_total][T] log2-domain shift of each token's tile
  float* part_s;  // [n_col_tiles_total][T] sum of 2^(z log2 e - shift) over the tile
  float* part_s2; // [n_col_tiles_total][T] (EPI_PARTIALS_ENT) sum of 2^(z log2 e - shift) z
  float* zy;      // [T] target logit
  const float* lse2;  // [T] LSE * log2(e)
  const float* coef;  // [T] gradient coefficient (grad scale included)
  // with the entropy bonus (eb != NULL): dz_v = p_v (ea + eb z_v) - coef [v == y]
  const float* ea;    // [T] coef - eb E_p[z]
  const float* eb;    // [T] entropy coefficient times the token's grad scale
  __nv_bfloat16* dz;  // chunk buffer [T][ldz], column 0 = vocabulary column v0
  int64_t ldz, v0;
  // EPI_STORE_F32: C[M][ldc] = (accumulate ? C : 0) + A B
  float* C;
  int64_t ldc;
  int accumulate;
  grpo_step_acc* acc;
  // A compact order of the tokens that the partition kernel wrote earlier in stream order:
  // *live_n of them, row i of the compact order being token row_idx[i]. The backward runs
  // over the live tokens (a dlogits row that is not all zero); pass A, when asked to skip the
  // masked tokens, over the valid ones. live_mode says which extent follows from the device
  // count (M and K above then give the allocated token rows, T):
  //   LIVE_ROWS_PADDED  rows = live tokens, and the epilogue writes zero dlogits rows up to the
  //                     padded count (live_pad below), so that dW's reduction over the padded
  //                     count reads zeros past the live rows;
  //   LIVE_ROWS         rows = live tokens (d_h: rows scattered to C[row_idx[i]]; pass A:
  //                     partials at the compact row, the target logit at the token);
  //   LIVE_K            reduction length = the padded count (dW over the compact tokens).
  const int32_t* live_n;
  const int32_t* row_idx;
  int live_mode;
};

enum { LIVE_NONE = 0, LIVE_ROWS_PADDED = 1, LIVE_ROWS = 2, LIVE_K = 3 };

// The padded live count: a multiple of the K block (at least one block, so that dW always
// reduces over at least one block of zeros), at most the allocated rows rounded up.
__device__ __forceinline__ int64_t live_pad(int64_t n, int64_t rows) {
  const int64_t p = n < BK ? (int64_t)BK : (n + BK - 1) / BK * BK;
  const int64_t cap = (rows + BK - 1) / BK * BK;
  return p < cap ? p : cap;
}

// Work unit t -> (unit along M, tile along N).
__device__ __forceinline__ void unit_coords(const GemmArgs& g, int n_m, int t, int& mu, int& nu) {
  if (g.m_fast) {
    mu = t % n_m;
    nu = t / n_m;
  } else {
    nu = t % g.n_n;
    mu = t / g.n_n;
  }
}

// ---- epilogues: thread = one accumulator row (TMEM lane), 256 columns at taddr ---------------

// Softmax partials of one 256-column vocabulary tile: lazy online (shift, sum) in log2 units and
// the target logit if the tile holds it. Zero-filled columns past the vocabulary count as -inf.
__device__ __forceinline__ void epi_partials(const GemmArgs& g, uint32_t taddr, int64_t row, bool rok, int ct) {
  const int64_t c0 = (int64_t)ct * BN;
  // the token of this row (the compact order's, when the masked tokens are skipped); the
  // partials stay at the row, the target logit goes to the token
  const int64_t tok = (rok && g.row_idx) ? (int64_t)g.row_idx[row] : row;
  const int32_t y = rok ? g.target[tok] : -1;
  const bool own = y >= c0 && y < c0 + BN;
  MS acc{-INFINITY, 0.f};
  float zy = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    const int64_t cb = c0 + c * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (cb + i >= g.V) v[i] = -INFINITY;
    if (own && y >= cb && y < cb + 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (cb + i == y) zy = v[i];
    }
    lazy_online2<32>(acc, v);
  }
  if (rok) {
    g.part_m[(int64_t)ct * g.M + row] = acc.m;
    g.part_s[(int64_t)ct * g.M + row] = acc.s;
    if (own) g.zy[tok] = zy;
  }
}

// epi_partials with the entropy's third accumulator: (shift, sum e, sum e z) of the tile, the
// target logit. Groups of 32 columns wholly past the vocabulary are skipped; a group holding
// both takes the no-mass guard for its -inf columns.
__device__ __forceinline__ void epi_partials_ent(const GemmArgs& g, uint32_t taddr, int64_t row, bool rok, int ct) {
  const int64_t c0 = (int64_t)ct * BN;
  const int64_t tok = (rok && g.row_idx) ? (int64_t)g.row_idx[row] : row;
  const int32_t y = rok ? g.target[tok] : -1;
  const bool own = y >= c0 && y < c0 + BN;
  MS3 acc{-INFINITY, 0.f, 0.f};
  bool guarded = false;
  float zy = 0.f;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    const int64_t cb = c0 + c * 32;
    if (cb >= g.V) continue;  // warp-uniform
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (cb + i >= g.V) v[i] = -INFINITY;
    if (own && y >= cb && y < cb + 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (cb + i == y) zy = v[i];
    }
    lazy_online3<32>(acc, v, guarded);
  }
  if (rok) {
    g.part_m[(int64_t)ct * g.M + row] = acc.m;
    g.part_s[(int64_t)ct * g.M + row] = acc.s;
    g.part_s2[(int64_t)ct * g.M + row] = acc.s2;
    if (own) g.zy[tok] = zy;
  }
}

// dlogits of one tile: dz = coef * 2^(z log2 e - LSE2) - coef [v == y], rounded to bf16 (|coef|
// is folded into the exponent, its sign applied to the packed pair). Masked and clipped tokens
// (coef = 0) give zero rows. Each 32-column group of the warp's 32 rows is staged in shared
// memory (64-byte swizzle: chunk q of row r at q ^ ((r >> 1) & 3), conflict-free for the
// warp's 16-byte writes) and written by one TMA store through map_c, whose extents (the chunk's
// vocabulary columns, T rows) clip the vocabulary tail and the rows past T.
__device__ __forceinline__ void epi_dlogits(const GemmArgs& g, const CUtensorMap* map_c, uint32_t taddr,
                                            int64_t row, bool rok, int ct, int64_t warp_row0, int64_t rows_store,
                                            uint32_t stage_buf, int lane) {
  const int64_t c0 = (int64_t)ct * BN;
  // the token of this accumulator row (the compact order's, in the live-token backward)
  const int64_t tok = (rok && g.row_idx) ? (int64_t)g.row_idx[row] : row;
  const int32_t y = rok ? g.target[tok] : -1;
  const float cf = rok ? g.coef[tok] : 0.f;
  const float l2 = rok ? g.lse2[tok] : 0.f;
  const float cexp = l2 - log2f(fabsf(cf));
  const uint32_t sgn = cf < 0.f ? 0x80008000u : 0u;
  // with the entropy bonus: dz = p (ea + eb z); ea = eb = 0 for masked tokens
  const bool ent = g.eb != nullptr;
  const float ea = (ent && rok) ? g.ea[tok] : 0.f, eb = (ent && rok) ? g.eb[tok] : 0.f;
  const bool live = ent ? (ea != 0.f || eb != 0.f) : cf != 0.f;
  const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    const int64_t cb = c0 + c * 32;
    // warp-uniform: the rest of the tile lies past the vocabulary, or all 32 rows past the
    // rows to be written (T, or the padded live count; rows in between get zeros)
    if (cb >= g.V || warp_row0 >= rows_store) continue;
    uint32_t w[16];
    if (live) {
      float zyv = 0.f;
      const bool hit = y >= cb && y < cb + 32;
      if (hit) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (cb + i == y) zyv = v[i];
      }
      if (ent) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 p = ex2_pair(v[i], v[i + 1], l2);
          w[i / 2] = pack_bf16x2(p.x * fmaf(eb, v[i], ea), p.y * fmaf(eb, v[i + 1], ea));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 p = ex2_pair(v[i], v[i + 1], cexp);
          w[i / 2] = pack_bf16x2(p.x, p.y) ^ sgn;
        }
      }
      if (hit) {
        const float py = ex2(fmaf(zyv, kLog2e, -l2));
        const float dzy = ent ? py * fmaf(eb, zyv, ea) - cf : cf * py - cf;
        const uint32_t hb = __bfloat16_as_ushort(__float2bfloat16_rn(dzy));
        const int k = (int)(y - cb);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (k == 2 * i) w[i] = (w[i] & 0xFFFF0000u) | hb;
          if (k == 2 * i + 1) w[i] = (w[i] & 0x0000FFFFu) | (hb << 16);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
    const uint32_t buf = stage_buf + (uint32_t)(c & 1) * EPI_BUF_BYTES;
    if (lane == 0) bulk_wait_read<1>();  // the store issued from this buffer two groups ago has read it
    __syncwarp();
    const uint32_t rb = buf + (uint32_t)lane * 64u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + (((uint32_t)q ^ sw) << 4)),
                   "r"(w[4 * q]), "r"(w[4 * q + 1]), "r"(w[4 * q + 2]), "r"(w[4 * q + 3])
                   : "memory");
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store2d(map_c, buf, (int)(cb - g.v0), (int)warp_row0);
      bulk_commit();
    }
  }
}

// float32 output tile: C[row][n0 .. n0 + 256) = (accumulate ? C : 0) + D, columns past N skipped
// (N is a multiple of 64, so a 32-column group is wholly inside or outside).
__device__ __forceinline__ void epi_store_f32(const GemmArgs& g, uint32_t taddr, int64_t row, bool rok, int64_t n0) {
  // d_h over the live tokens: compact row -> the token's row of C
  const int64_t crow_i = (rok && g.row_idx) ? (int64_t)g.row_idx[row] : row;
  float* crow = g.C + crow_i * g.ldc;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + c * 32, v);
    const int64_t col = n0 + c * 32;
    if (!rok || col >= g.N) continue;
    float4* p = reinterpret_cast<float4*>(crow + col);
    if (g.accumulate) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 o = p[q];
        v[4 * q] += o.x;
        v[4 * q + 1] += o.y;
        v[4 * q + 2] += o.z;
        v[4 * q + 3] += o.w;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

// ---- the kernel ---------------------------------------------------------------------------------

template <int CG, int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NTHREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
            const __grid_constant__ CUtensorMap map_c, GemmArgs g) {
  using S = Shape<CG, EPI>;
  constexpr uint32_t ID = idesc<CG, A_MN, B_MN>();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t epi_base = sbase + S::STAGES * S::STAGE_BYTES;  // dlogits staging (1024-aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(sgen + S::STAGES * S::STAGE_BYTES + S::EPI_BYTES);
  uint64_t* empty = full + S::STAGES;
  uint64_t* tfull = empty + S::STAGES;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * CG);  // every epilogue warp of the cluster releases the buffer
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<CG>(smem_u32(tmem_slot));  // with CG = 2 one warp of each CTA
  fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync_all();  // the peer's barriers exist before anything targets them
  fence_after();
  const uint32_t tmem = *tmem_slot;

  // extents: the launch's, or, in the live-token backward, from the device count (written by
  // an earlier kernel in stream order; every thread reads the same value)
  int64_t M = g.M, rows_store = g.M, K = g.K;
  int n_m = g.n_m;
  if (g.live_mode != LIVE_NONE) {
    const int64_t nl = *g.live_n;
    if (g.live_mode == LIVE_K) {
      K = live_pad(nl, g.K);
    } else {
      M = nl;
      rows_store = g.live_mode == LIVE_ROWS_PADDED ? live_pad(nl, g.M) : nl;
      if (rows_store > g.M) rows_store = g.M;
      n_m = (int)((rows_store + BM * CG - 1) / (BM * CG));
    }
  }
  const int n_units = n_m * g.n_n;
  const int first = CG == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int stride = CG == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int KB = (int)((K + BK - 1) / BK);

  if (warp == 0) {
    // ---- TMA producer: this CTA's A rows and B rows of every stage ----
    if (lane == 0) {
      const uint32_t full0 = CG == 2 ? mapa_u32(smem_u32(full), 0) : smem_u32(full);
      uint32_t stage = 0, phase = 0;
      for (int t = first; t < n_units; t += stride) {
        int mu, nu;
        unit_coords(g, n_m, t, mu, nu);
        const int a_row = mu * BM * CG + (int)rank * BM;
        const int b_row = (g.col_tile0 + nu) * BN + (int)rank * S::B_ROWS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, s_abort)) break;
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], CG * S::STAGE_BYTES);
          const uint32_t sa = sbase + stage * S::STAGE_BYTES;
          const uint32_t bar = full0 + stage * 8u;
          load_operand<CG, A_MN, BM>(sa, &map_a, bar, kb * BK, a_row);
          load_operand<CG, B_MN, S::B_ROWS>(sa + S::A_BYTES, &map_b, bar, kb * BK, b_row);
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (*s_abort) break;  // a wait gave up: issue nothing more
      }
      // every stage's last release has arrived before this CTA may leave: the MMAs that read
      // this CTA's shared memory are complete and no commit still targets its barriers
      for (int i = 0; i < S::STAGES; ++i) {  // a stage never used passes at once
        if (*s_abort)
          drain_wait(&empty[stage], phase ^ 1u);
        else
          mbar_wait_bounded(&empty[stage], phase ^ 1u, s_abort);
        if (++stage == S::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (the cluster's even CTA) ----
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, ab = 0, aphase = 0;
      for (int t = first; t < n_units; t += stride) {
        // the even CTA waits for both CTAs' epilogues to have read the accumulator (their
        // arrives release the TMEM reads at cluster scope)
        const bool free_acc = CG == 2 ? mbar_wait_cluster_bounded(&tempty[ab], aphase ^ 1u, s_abort)
                                      : mbar_wait_bounded(&tempty[ab], aphase ^ 1u, s_abort);
        if (!free_acc) break;
        fence_after();
        const uint32_t d = tmem + ab * BN;
        for (int kb = 0; kb < KB; ++kb) {
          // Not tested for a break: after a wait gives up, the unit's remaining MMAs issue
          // without waiting (they read whatever the stages hold; the step is flagged) and the
          // abort check below stops the issuer before the accumulator is committed. A break
          // here left the tensor pipe busy 88% of active cycles in pass A instead of 99%.
          mbar_wait_bounded(&full[stage], phase, s_abort);
          fence_after();
          const uint32_t sa = sbase + stage * S::STAGE_BYTES;
          const uint64_t da = sdesc<A_MN>(sa), db = sdesc<B_MN>(sa + S::A_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)
            mma_bf16<CG>(d, da + kstep<A_MN>() * j, db + kstep<B_MN>() * j, ID, kb > 0 || j > 0);
          const uint32_t eb = smem_u32(&empty[stage]);
          mma_commit<CG>(eb);
          if (CG == 2) mma_commit<CG>(mapa_u32(eb, 1));
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (*s_abort) break;  // the epilogues' waits give up on their own
        const uint32_t fb = smem_u32(&tfull[ab]);
        mma_commit<CG>(fb);
        if (CG == 2) mma_commit<CG>(mapa_u32(fb, 1));
        if (++ab == 2) {
          ab = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // ---- epilogue: warps 2..5, thread = TMEM lane = accumulator row ----
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may access
    const int trow = quarter * 32 + lane;
    uint32_t ab = 0, aphase = 0;
    for (int t = first; t < n_units; t += stride) {
      int mu, nu;
      unit_coords(g, n_m, t, mu, nu);
      mbar_wait_bounded(&tfull[ab], aphase, s_abort);
      fence_after();
      const int64_t row = (int64_t)mu * BM * CG + (int64_t)rank * BM + trow;
      const bool rok = row < M;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + ab * BN;
      if constexpr (EPI == EPI_PARTIALS)
        epi_partials(g, taddr, row, rok, g.col_tile0 + nu);
      else if constexpr (EPI == EPI_PARTIALS_ENT)
        epi_partials_ent(g, taddr, row, rok, g.col_tile0 + nu);
      else if constexpr (EPI == EPI_DLOGITS)
        epi_dlogits(g, &map_c, taddr, row, rok, g.col_tile0 + nu, row - lane, rows_store,
                    epi_base + (uint32_t)quarter * 2u * EPI_BUF_BYTES, lane);
      else
        epi_store_f32(g, taddr, row, rok, (int64_t)nu * BN);
      fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2 && rank != 0)
          mbar_arrive_remote(mapa_u32(smem_u32(&tempty[ab]), 0));
        else
          mbar_arrive(&tempty[ab]);
      }
      if (++ab == 2) {
        ab = 0;
        aphase ^= 1u;
      }
    }
    if (EPI == EPI_DLOGITS && lane == 0) bulk_wait_all();  // this warp's stores are complete
  }

  fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync_all();  // neither CTA leaves while the other may still signal it
  if (*s_abort && threadIdx.x == 0) atomicOr(&g.acc->flags, kFlagWaitTimeout);
  if (warp == 1) {
    fence_after();
    tmem_dealloc<CG>(tmem);
  }
}

}  // namespace lmhead
}  // namespace grpo
