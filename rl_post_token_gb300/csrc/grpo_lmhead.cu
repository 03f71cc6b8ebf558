// Fused LM-head variant of the loss: the logits z = h W^T are produced on the tensor cores
// tile by tile and consumed by the softmax in the GEMM epilogue, so the [T, V] float32 logits
// and their softmax never reach memory ("Sizing mini-batches and micro-batches", "The problem":
// the log-softmax over the vocabulary of 2048-token completions is what runs out of memory).
//
//  pass A  tcgen05 GEMM over all (128-token x 256-vocab) tiles; the epilogue reduces each
//          tile row to a log2-domain (shift, sum-exp) partial and picks up the target logit
//          (stored path: it also writes e = 2^(z log2 e - shift) of the tile as bf16).
//  reduce  per token: combine the partials in vocabulary order -> LSE, log-prob, ratio,
//          clipped surrogate, gradient coefficient (same token epilogue as the row pass).
//  backward, recompute path (minimum workspace): per vocabulary chunk the same GEMM recomputes
//          the chunk's logits and its epilogue writes dlogits (bf16) into a bounded chunk
//          workspace; then d_h += dz_c W_c and dW_c = dz_c^T h (cuBLAS, float32 outputs).
//  backward, stored path (workspace for the whole [T, V] exponent matrix): dz_from_e_kernel
//          turns the stored e into dlogits in place; then one d_h and one dW GEMM.
//
// GEMM kernel: persistent, one CTA per SM, 6 warps, launched as 2-CTA clusters (CTA pair) or
// as single CTAs. Warp 0 issues TMA loads (128-byte swizzled 128x64 h tiles and 256x64 W tiles;
// in a pair each CTA loads one 128-row half of W, multicast to both) into a 4-stage
// shared-memory ring; warp 1 issues tcgen05.mma (M=128, N=256, K=16, bf16 -> f32) into a
// double-buffered TMEM accumulator (2 x 256 columns); warps 2-5 read the accumulator with
// tcgen05.ld (one TMEM lane = one token row per thread) and run the epilogue while the next
// tile's MMAs proceed. Every mbarrier wait is bounded and raises a flag instead of hanging.
#include <cublas_v2.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "grpo_common.cuh"

namespace grpo {
namespace lmhead {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NTHREADS = 192;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr size_t SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + 256;

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16, both K-major,
// N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle: rows of 128 bytes,
// 8-row swizzle atoms 1024 bytes apart (stride byte offset), version 1, layout SWIZZLE_128B.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, bool accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(kIdesc), "r"((uint32_t)accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// CTA-pair variants: the load lands at the same shared-memory offset in every CTA of `mask`
// and completes bytes on the mbarrier at `bar`'s offset in each of them; the commit arrives on
// the mbarrier at `bar`'s offset in every CTA of `mask`.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(bar), "h"(mask)
      : "memory");
}

// Bounded wait that ignores the abort flag: the end-of-kernel drains after a timeout.
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
  int64_t T, V, H;
  int n_row_tiles;
  int col_tile0, n_col_tiles;  // tiles [col_tile0, col_tile0 + n_col_tiles) of 256 columns
  int mode;                    // 0: softmax partials; 1: dlogits
  const int32_t* target;
  // mode 0
  float* part_m;  // [n_col_tiles_total][T] log2-domain max
  float* part_s;  // [n_col_tiles_total][T]
  float* zy;      // [T] target logit
  // mode 0 with est != NULL: e = 2^((z - tile max) log2 e) stored as bf16 [T][lde] (the
  // partials then use the exact tile maximum)
  __nv_bfloat16* est;
  int64_t lde;
  // mode 1
  const float* lse2;  // [T] LSE * log2(e)
  const float* coef;  // [T] gradient coefficient (already scaled)
  __nv_bfloat16* dz;  // chunk workspace [T][ldz], column 0 = vocabulary column v0
  int64_t ldz, v0;
  grpo_step_acc* acc;
};

// Stored path: e = 2^(z log2 e - shift) of 32 columns (-inf past the vocabulary gives 0),
// written as bf16 for row `row` (if it exists) and added to s.
__device__ __forceinline__ void store_e_chunk(const GemmArgs& g, bool rok, int64_t row, int64_t cb, float (&v)[32],
                                              float shift, float& s) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = ex2(fmaf(v[i], kLog2e, -shift));
  if (rok) {
    uint4* d4 = reinterpret_cast<uint4*>(g.est + row * g.lde + cb);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      d4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                         pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  }
  s += tree_sum(v);  // reduces v in place: after the store
}

// Work units of a launch. One CTA: a unit is one 128 x 256 tile. CTA pair (a 2-CTA cluster): a
// unit is two vertically adjacent tiles sharing one W tile; CTA r of the pair computes row tile
// 2u + r (past the last row tile it computes zero-filled rows whose results are discarded).
template <bool PAIR>
struct Units {
  int n_row_units, n, first, stride;
  uint32_t rank;
  __device__ Units(const GemmArgs& g, uint32_t r) : rank(r) {
    n_row_units = PAIR ? (g.n_row_tiles + 1) / 2 : g.n_row_tiles;
    n = n_row_units * g.n_col_tiles;
    first = PAIR ? (int)(blockIdx.x / 2) : (int)blockIdx.x;
    stride = PAIR ? (int)(gridDim.x / 2) : (int)gridDim.x;
  }
  __device__ void tile(const GemmArgs& g, int t, int& rt, int& ct) const {
    const int ru = t % n_row_units;
    ct = g.col_tile0 + t / n_row_units;
    rt = PAIR ? 2 * ru + (int)rank : ru;
  }
};

// PAIR = false: one CTA per SM loads its h tile and the whole W tile. PAIR = true: the two CTAs
// of a cluster each load their own h tile and one 128-row half of the shared W tile, multicast
// into both, so each CTA pulls 32 KB per K step from L2 instead of 48 KB. A stage is refilled
// only after both CTAs' MMAs have released it (each commit arrives on both CTAs' barrier).
template <bool PAIR>
__global__ void __launch_bounds__(NTHREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w, GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  uint64_t* full = reinterpret_cast<uint64_t*>(sgen + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAIR ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the peer's barriers exist before anything targets them
  fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const Units<PAIR> units(g, rank);
  const int KB = (int)(g.H / BK);
  uint32_t issued = 0;  // producer: stage loads issued

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int t = units.first; t < units.n; t += units.stride) {
        int rt, ct;
        units.tile(g, t, rt, ct);
        for (int kb = 0; kb < KB; ++kb) {
          mbar_wait_bounded(&empty[stage], phase ^ 1u, s_abort);
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          tma_load_2d(sa, &map_h, smem_u32(&full[stage]), kb * BK, rt * BM);
          if (PAIR)
            tma_load_2d_mc(sa + A_BYTES + rank * (B_BYTES / 2), &map_w, smem_u32(&full[stage]), kb * BK,
                           ct * BN + (int)rank * (BN / 2), (uint16_t)0x3);
          else
            tma_load_2d(sa + A_BYTES, &map_w, smem_u32(&full[stage]), kb * BK, ct * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (PAIR) {
        // every stage's last release (this CTA's commit and the peer's) has arrived before
        // this CTA may leave: the peer's commits target this CTA's barriers
        for (int i = 0; i < STAGES; ++i) {  // a stage never used passes at once
          mbar_wait_bounded(&empty[stage], phase ^ 1u, s_abort);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, ab = 0, aphase = 0;
      for (int t = units.first; t < units.n; t += units.stride) {
        mbar_wait_bounded(&tempty[ab], aphase ^ 1u, s_abort);
        fence_after();
        const uint32_t d = tmem + ab * BN;
        for (int kb = 0; kb < KB; ++kb) {
          mbar_wait_bounded(&full[stage], phase, s_abort);
          fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + A_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)  // +32 bytes along K per 16-element step
            mma_bf16(d, da + 2 * j, db + 2 * j, kb > 0 || j > 0);
          if (PAIR)
            mma_commit_mc(smem_u32(&empty[stage]), (uint16_t)0x3);
          else
            mma_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        mma_commit(smem_u32(&tfull[ab]));
        if (++ab == 2) {
          ab = 0;
          aphase ^= 1u;
        }
      }
    }
  } else {
    // ---- epilogue: warps 2..5, thread = TMEM lane = token row of the tile ----
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int trow = quarter * 32 + lane;
    uint32_t ab = 0, aphase = 0;
    for (int t = units.first; t < units.n; t += units.stride) {
      int rt, ct;
      units.tile(g, t, rt, ct);
      mbar_wait_bounded(&tfull[ab], aphase, s_abort);
      fence_after();
      const int64_t row = (int64_t)rt * BM + trow;
      const int64_t c0 = (int64_t)ct * BN;
      const bool rok = row < g.T;
      const int32_t y = rok ? g.target[row] : -1;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + ab * BN;
      if (g.mode == 0 && g.est) {
        // one pass: e relative to a shift taken from the first 32 columns, stored and summed;
        // if a later value sits more than 2^64 above that shift the warp redoes the tile
        // with the exact tile maximum (e <= 2^64 keeps every stored value and the sum finite)
        float shift = 0.f, s = 0.f, zy = 0.f;
        bool redo = false;
        const bool own = y >= c0 && y < c0 + BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int64_t cb = c0 + c * 32;
          float cmax = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (cb + i >= g.V) v[i] = -INFINITY;
            cmax = fmaxf(cmax, v[i]);
          }
          if (own && y >= cb && y < cb + 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i == y) zy = v[i];
          }
          if (c == 0) shift = cmax * kLog2e;  // the first 32 columns always hold vocabulary entries
          redo |= !(cmax * kLog2e <= shift + 64.f);
          store_e_chunk(g, rok, row, cb, v, shift, s);
        }
        if (__any_sync(0xffffffffu, redo)) {
          float mx = -INFINITY;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            const int64_t cb = c0 + c * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i < g.V) mx = fmaxf(mx, v[i]);
          }
          shift = mx * kLog2e;
          s = 0.f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            const int64_t cb = c0 + c * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i >= g.V) v[i] = -INFINITY;
            store_e_chunk(g, rok, row, cb, v, shift, s);
          }
        }
        if (rok) {
          g.part_m[(int64_t)ct * g.T + row] = shift;
          g.part_s[(int64_t)ct * g.T + row] = s;
          if (own) g.zy[row] = zy;
        }
      } else if (g.mode == 0) {
        MS acc{-INFINITY, 0.f};
        float zy = 0.f;
        const bool own = y >= c0 && y < c0 + BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int64_t cb = c0 + c * 32;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (cb + i >= g.V) v[i] = -INFINITY;  // zero-filled columns past the vocabulary
          if (own && y >= cb && y < cb + 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cb + i == y) zy = v[i];
          }
          lazy_online2<32>(acc, v);
        }
        if (rok) {
          g.part_m[(int64_t)ct * g.T + row] = acc.m;
          g.part_s[(int64_t)ct * g.T + row] = acc.s;
          if (own) g.zy[row] = zy;
        }
      } else {
        const float cf = rok ? g.coef[row] : 0.f;
        const float l2 = rok ? g.lse2[row] : 0.f;
        const float cexp = l2 - log2f(fabsf(cf));
        const uint32_t sgn = cf < 0.f ? 0x80008000u : 0u;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int64_t cb = c0 + c * 32;
          if (!rok || cb >= g.V) continue;
          uint32_t w[16];
          if (cf != 0.f) {
            float zyv = 0.f;
            const bool hit = y >= cb && y < cb + 32;
            if (hit) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (cb + i == y) zyv = v[i];
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = ex2(fmaf(v[i], kLog2e, -cexp));
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]) ^ sgn;
            if (hit) {
              const float dzy = cf * ex2(fmaf(zyv, kLog2e, -l2)) - cf;
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
          __nv_bfloat16* dst = g.dz + row * g.ldz + (cb - g.v0);
          const int nvalid = (int)std::min<int64_t>(32, g.V - cb);
          if (nvalid == 32) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int q = 0; q < 4; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          } else {
            for (int i = 0; i < nvalid; ++i)
              dst[i] = __ushort_as_bfloat16((unsigned short)((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu)));
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[ab]);
      if (++ab == 2) {
        ab = 0;
        aphase ^= 1u;
      }
    }
  }

  fence_before();
  __syncthreads();
  if (PAIR) {
    cluster_sync_all();  // neither CTA leaves while the other may still signal or copy into it
    if (*s_abort && threadIdx.x == 0) {
      // after a timeout, let this CTA's copies and the peer's arrivals settle (bounded)
      for (int sidx = 0; sidx < STAGES && (uint32_t)sidx < issued; ++sidx) {
        const uint32_t uses = (issued - 1u - (uint32_t)sidx) / STAGES;
        drain_wait(&full[sidx], uses & 1u);
        drain_wait(&empty[sidx], uses & 1u);
      }
    }
  }
  if (*s_abort && threadIdx.x == 0) atomicOr(&g.acc->flags, kFlagWaitTimeout);
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// Per token: combine the vocabulary-tile partials in order, then the token epilogue.
__global__ void reduce_kernel(int64_t T, int n_col_tiles, const float* __restrict__ part_m,
                              const float* __restrict__ part_s, const float* __restrict__ zy,
                              const int32_t* __restrict__ target, int64_t V, const float* old_logp,
                              const float* __restrict__ adv, const uint8_t* __restrict__ mask, float eps,
                              float scale, float* __restrict__ lse2_out, float* __restrict__ coef_out,
                              float* loss_tok, float* logp_tok, grpo_step_acc* acc) {
  __shared__ unsigned long long sc[4];
  if (threadIdx.x < 4) sc[threadIdx.x] = 0;
  __syncthreads();
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned long long v_valid = 0, v_clip = 0, v_nf = 0, v_tok = 0;
  if (row < T) {
    v_tok = 1;
    float coef = 0.f, l2 = 0.f;
    if (mask[row]) {
      MS t{-INFINITY, 0.f};
      for (int c = 0; c < n_col_tiles; ++c) t = ms2_combine(t, MS{part_m[(int64_t)c * T + row], part_s[(int64_t)c * T + row]});
      const float l2s = log2f(t.s);
      l2 = t.m + l2s;
      const int32_t y = target[row];
      const float z = (y >= 0 && (int64_t)y < V) ? zy[row] : __int_as_float(0x7fc00000);
      // log2 p_y = (z_y log2e - m) - log2(sum), without cancellation
      const TokenOut o = token_epilogue((fmaf(z, kLog2e, -t.m) - l2s) * kLn2, fabsf(l2) <= kLseMax * kLog2e,
                                        old_logp != nullptr, old_logp ? old_logp[row] : 0.f, adv[row], eps, scale);
      loss_tok[row] = o.loss;
      if (logp_tok) logp_tok[row] = o.logp;
      coef = o.coef;
      v_valid = 1;
      v_clip = o.clipped;
      v_nf = o.nonfinite;
    } else {
      loss_tok[row] = 0.f;
      if (logp_tok) logp_tok[row] = 0.f;
    }
    lse2_out[row] = l2;
    coef_out[row] = coef;
  }
  if (v_tok) atomicAdd(&sc[0], v_tok);
  if (v_valid) atomicAdd(&sc[1], v_valid);
  if (v_clip) atomicAdd(&sc[2], v_clip);
  if (v_nf) atomicAdd(&sc[3], v_nf);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sc[0]) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_tokens), sc[0]);
    if (sc[1]) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_valid), sc[1]);
    if (sc[2]) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_clipped), sc[2]);
    if (sc[3]) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_nonfinite), sc[3]);
  }
}

// Stored path, backward: dz = coef * 2^(tile max - LSE) * e, in place over the stored e, one CTA
// per token row at a time; the target element, coef * (p_y - 1), is taken from the float32
// target logit and written by the thread that wrote its vector.
__global__ void __launch_bounds__(256) dz_from_e_kernel(int64_t T, int64_t V, int n_col_tiles, int64_t lde,
                                                        const float* __restrict__ part_m,
                                                        const float* __restrict__ lse2,
                                                        const float* __restrict__ coef,
                                                        const float* __restrict__ zy,
                                                        const int32_t* __restrict__ target,
                                                        __nv_bfloat16* __restrict__ e) {
  extern __shared__ float f[];  // [n_col_tiles] per-tile factor of the current row
  const int tid = threadIdx.x;
  const int64_t nv = lde / 8;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const float c = coef[row], l2 = lse2[row];
    __syncthreads();
    for (int ct = tid; ct < n_col_tiles; ct += blockDim.x)
      f[ct] = c == 0.f ? 0.f : c * ex2(part_m[(int64_t)ct * T + row] - l2);
    __syncthreads();
    uint4* p = reinterpret_cast<uint4*>(e + row * lde);
    if (c == 0.f) {  // masked or clipped: a zero row, whatever e holds
      for (int64_t v = tid; v < nv; v += blockDim.x) p[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    for (int64_t v = tid; v < nv; v += blockDim.x) {
      const float fv = f[v / (BN / 8)];
      uint4 u = p[v];
      float x[8];
      x[0] = bf16_lo(u.x) * fv; x[1] = bf16_hi(u.x) * fv; x[2] = bf16_lo(u.y) * fv; x[3] = bf16_hi(u.y) * fv;
      x[4] = bf16_lo(u.z) * fv; x[5] = bf16_hi(u.z) * fv; x[6] = bf16_lo(u.w) * fv; x[7] = bf16_hi(u.w) * fv;
      p[v] = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                        pack_bf16x2(x[6], x[7]));
    }
    const int32_t y = target[row];
    if (y >= 0 && (int64_t)y < V && tid == (int)((y / 8) % blockDim.x))
      e[row * lde + y] = __float2bfloat16_rn(c * ex2(fmaf(zy[row], kLog2e, -l2)) - c);
  }
}

// ---- host -------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, cols] bf16 matrix, box [box_rows, 64] with 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The current device's cuBLAS handle, created on first use. A handle's stream and workspace
// are settings of the handle, so the caller holds `lock` (taken here) from setting them until
// its last GEMM is enqueued: calls from several host threads then never enqueue on one
// another's stream or scratch.
cublasHandle_t blas_handle(std::unique_lock<std::mutex>& lock) {
  static cublasHandle_t h[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  lock = std::unique_lock<std::mutex>(mu);
  if (!h[dev] && cublasCreate(&h[dev]) != CUBLAS_STATUS_SUCCESS) h[dev] = nullptr;
  return h[dev];
}

// GEMM variant: the CTA pair unless GRPO_LMHEAD_PAIR=0 selects the one-CTA kernel.
bool use_pair() {
  const char* e = getenv("GRPO_LMHEAD_PAIR");
  return !(e && e[0] == '0');
}

// h and W tensor maps for a variant (the pair loads W in 128-row halves).
bool make_maps(CUtensorMap* map_h, CUtensorMap* map_w, const void* h, const void* W, int64_t T, int64_t V, int64_t H,
               bool pair) {
  return make_map(map_h, h, (uint64_t)T, (uint64_t)H, BM) &&
         make_map(map_w, W, (uint64_t)V, (uint64_t)H, pair ? BN / 2 : BN);
}

// Launch one GEMM pass over the tiles g describes. The first launch of a variant on a device
// sets its shared-memory limit and caches how many CTAs (or CTA pairs) fit at once.
template <bool PAIR>
int launch_gemm_t(const CUtensorMap& map_h, const CUtensorMap& map_w, const GemmArgs& g, cudaStream_t st) {
  auto kern = gemm_kernel<PAIR>;
  int dev = 0;
  GRPO_CUDA_TRY(cudaGetDevice(&dev));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 1 : 0;
  int max_units = 0;
  {
    static std::mutex mu;
    static int cached[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64) max_units = cached[dev];
    if (max_units == 0) {
      GRPO_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES));
      if (PAIR) {
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        GRPO_CUDA_TRY(cudaOccupancyMaxActiveClusters(&max_units, kern, &cfg));
      } else {
        max_units = sm_count();
      }
      if (max_units < 1) return GRPO_ERR_UNSUPPORTED;
      if (dev >= 0 && dev < 64) cached[dev] = max_units;
    }
  }
  const int64_t row_units = PAIR ? (g.n_row_tiles + 1) / 2 : g.n_row_tiles;
  const int64_t units = std::min<int64_t>(row_units * g.n_col_tiles, max_units);
  if (units <= 0) return GRPO_OK;
  cfg.gridDim = dim3((unsigned)(PAIR ? 2 * units : units), 1, 1);
  GRPO_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, map_h, map_w, g));
  return GRPO_OK;
}

int launch_gemm(bool pair, const CUtensorMap& map_h, const CUtensorMap& map_w, const GemmArgs& g, cudaStream_t st) {
  return pair ? launch_gemm_t<true>(map_h, map_w, g, st) : launch_gemm_t<false>(map_h, map_w, g, st);
}

}  // namespace lmhead
}  // namespace grpo

using namespace grpo;
using namespace grpo::lmhead;

namespace {

// Scratch of the backward GEMMs, a region of the caller's workspace: each call brings its own,
// so GEMMs of calls that overlap on several streams share none.
constexpr size_t kBlasWorkspaceBytes = (size_t)32 << 20;

struct WsLayout {
  size_t part_m, part_s, zy, lse2, coef, dz, blas, total;
  int n_col_tiles;
  int64_t vchunk;  // columns of the dz region: one recompute chunk, or (stored) every tile
};

// stored = true: the dz region holds the whole [T, n_col_tiles * 256] exponent/dlogits matrix
WsLayout ws_layout(int64_t T, int64_t V, int64_t vchunk, bool stored = false) {
  WsLayout w{};
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w.n_col_tiles = (int)((V + BN - 1) / BN);
  w.vchunk = stored ? (int64_t)w.n_col_tiles * BN : std::min<int64_t>(vchunk, (int64_t)w.n_col_tiles * BN);
  size_t off = 0;
  w.part_m = off; off += up((size_t)w.n_col_tiles * T * 4);
  w.part_s = off; off += up((size_t)w.n_col_tiles * T * 4);
  w.zy = off; off += up((size_t)T * 4);
  w.lse2 = off; off += up((size_t)T * 4);
  w.coef = off; off += up((size_t)T * 4);
  w.dz = off; off += up((size_t)T * w.vchunk * 2);
  w.blas = off; off += kBlasWorkspaceBytes;
  w.total = off;
  return w;
}

constexpr int64_t kDefaultVChunk = 16384;  // vocabulary columns per pass-B chunk (64 tiles)

}  // namespace

extern "C" GRPO_API size_t grpo_lmhead_workspace_size(int64_t T, int64_t V, int64_t H) {
  if (T <= 0 || V <= 0 || H <= 0) return 0;
  return ws_layout(T, V, kDefaultVChunk).total;
}

extern "C" GRPO_API size_t grpo_lmhead_workspace_size_stored(int64_t T, int64_t V, int64_t H) {
  if (T <= 0 || V <= 0 || H <= 0) return 0;
  return ws_layout(T, V, kDefaultVChunk, true).total;
}

extern "C" GRPO_API int grpo_lmhead_loss_fwd_bwd(const void* h, const void* W, int64_t T, int64_t V, int64_t H,
                                                 const int32_t* target, const float* old_logp,
                                                 const float* adv_tok, const uint8_t* mask, float clip_eps,
                                                 float grad_scale, float* d_h, float* dW, float* loss_tok,
                                                 float* logp_tok, grpo_step_acc* acc, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
  if (T < 0 || V < 1 || H < BK || H % BK != 0 || !acc) return GRPO_ERR_INVALID;
  if (T == 0) return GRPO_OK;
  if (!h || !W || !target || !adv_tok || !mask || !loss_tok || !workspace) return GRPO_ERR_INVALID;
  if (((uintptr_t)h | (uintptr_t)W) & 15u) return GRPO_ERR_INVALID;
  if ((uintptr_t)workspace & 255u) return GRPO_ERR_INVALID;
  if (T > INT32_MAX / 2 || V > INT32_MAX / 2) return GRPO_ERR_INVALID;
  // the stored path when there is a backward pass and room for the whole exponent matrix
  const bool stored = (d_h || dW) && workspace_bytes >= ws_layout(T, V, kDefaultVChunk, true).total;
  const WsLayout ws = ws_layout(T, V, kDefaultVChunk, stored);
  if (workspace_bytes < ws.total) return GRPO_ERR_CAPACITY;
  const cudaStream_t st = as_stream(stream);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* part_m = reinterpret_cast<float*>(wsb + ws.part_m);
  float* part_s = reinterpret_cast<float*>(wsb + ws.part_s);
  float* zy = reinterpret_cast<float*>(wsb + ws.zy);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  float* coef = reinterpret_cast<float*>(wsb + ws.coef);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(wsb + ws.dz);

  const bool pair = use_pair();
  CUtensorMap map_h, map_w;
  if (!make_maps(&map_h, &map_w, h, W, T, V, H, pair)) return GRPO_ERR_UNSUPPORTED;
  const int n_row_tiles = (int)((T + BM - 1) / BM);

  GemmArgs g{};
  g.T = T;
  g.V = V;
  g.H = H;
  g.n_row_tiles = n_row_tiles;
  g.target = target;
  g.part_m = part_m;
  g.part_s = part_s;
  g.zy = zy;
  g.lse2 = lse2;
  g.coef = coef;
  g.dz = dz;
  g.ldz = ws.vchunk;
  g.acc = acc;
  g.est = stored ? dz : nullptr;
  g.lde = ws.vchunk;

  // pass A: softmax partials over every vocabulary tile
  g.mode = 0;
  g.col_tile0 = 0;
  g.n_col_tiles = ws.n_col_tiles;
  {
    const int rc = launch_gemm(pair, map_h, map_w, g, st);
    if (rc != GRPO_OK) return rc;
  }
  reduce_kernel<<<(unsigned)((T + 255) / 256), 256, 0, st>>>(T, ws.n_col_tiles, part_m, part_s, zy, target, V,
                                                              old_logp, adv_tok, mask, clip_eps, grad_scale, lse2,
                                                              coef, loss_tok, logp_tok, acc);
  GRPO_CUDA_TRY(cudaGetLastError());
  if (!d_h && !dW) return GRPO_OK;

  std::unique_lock<std::mutex> blas_lock;
  cublasHandle_t bh = blas_handle(blas_lock);
  if (!bh || cublasSetStream(bh, st) != CUBLAS_STATUS_SUCCESS ||
      cublasSetWorkspace(bh, wsb + ws.blas, kBlasWorkspaceBytes) != CUBLAS_STATUS_SUCCESS)
    return GRPO_ERR_CUDA;
  const float one = 1.f, zero = 0.f;
  if (stored) {
    // dlogits in place over the stored exponents, then each backward GEMM over the whole vocabulary
    const int grid = (int)std::min<int64_t>(T, (int64_t)sm_count() * 8);
    const size_t fsm = (size_t)ws.n_col_tiles * sizeof(float);
    if (fsm > 48 * 1024) return GRPO_ERR_UNSUPPORTED;
    dz_from_e_kernel<<<grid, 256, fsm, st>>>(T, V, ws.n_col_tiles, ws.vchunk, part_m, lse2, coef, zy, target, dz);
    GRPO_CUDA_TRY(cudaGetLastError());
    // d_h[T,H] = dz[T,V] W[V,H]   (column-major view: d_h^T = W^T dz^T)
    if (d_h && cublasGemmEx(bh, CUBLAS_OP_N, CUBLAS_OP_N, (int)H, (int)T, (int)V, &one, W, CUDA_R_16BF, (int)H, dz,
                            CUDA_R_16BF, (int)ws.vchunk, &zero, d_h, CUDA_R_32F, (int)H, CUBLAS_COMPUTE_32F,
                            CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return GRPO_ERR_CUDA;
    // dW[V,H] = dz^T[V,T] h[T,H]   (column-major view: dW^T = h^T dz)
    if (dW && cublasGemmEx(bh, CUBLAS_OP_N, CUBLAS_OP_T, (int)H, (int)V, (int)T, &one, h, CUDA_R_16BF, (int)H, dz,
                           CUDA_R_16BF, (int)ws.vchunk, &zero, dW, CUDA_R_32F, (int)H, CUBLAS_COMPUTE_32F,
                           CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return GRPO_ERR_CUDA;
    return GRPO_OK;
  }

  // recompute path: per vocabulary chunk, dlogits into the workspace, then the two backward GEMMs
  const int tiles_per_chunk = (int)(ws.vchunk / BN);
  for (int ct0 = 0, c = 0; ct0 < ws.n_col_tiles; ct0 += tiles_per_chunk, ++c) {
    const int nct = std::min(tiles_per_chunk, ws.n_col_tiles - ct0);
    const int64_t v0 = (int64_t)ct0 * BN;
    const int64_t vc = std::min<int64_t>((int64_t)nct * BN, V - v0);
    g.mode = 1;
    g.col_tile0 = ct0;
    g.n_col_tiles = nct;
    g.v0 = v0;
    const int rc = launch_gemm(pair, map_h, map_w, g, st);
    if (rc != GRPO_OK) return rc;
    const __nv_bfloat16* Wc = static_cast<const __nv_bfloat16*>(W) + v0 * H;
    // d_h[T,H] (+)= dz[T,vc] W_c[vc,H]   (column-major view: d_h^T = W_c^T dz^T)
    if (d_h &&
        cublasGemmEx(bh, CUBLAS_OP_N, CUBLAS_OP_N, (int)H, (int)T, (int)vc, &one, Wc, CUDA_R_16BF, (int)H, dz,
                     CUDA_R_16BF, (int)ws.vchunk, c == 0 ? &zero : &one, d_h, CUDA_R_32F, (int)H,
                     CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return GRPO_ERR_CUDA;
    // dW_c[vc,H] = dz^T[vc,T] h[T,H]   (column-major view: dW_c^T = h^T dz)
    if (dW && cublasGemmEx(bh, CUBLAS_OP_N, CUBLAS_OP_T, (int)H, (int)vc, (int)T, &one, h, CUDA_R_16BF, (int)H, dz,
                           CUDA_R_16BF, (int)ws.vchunk, &zero, dW + v0 * H, CUDA_R_32F, (int)H, CUBLAS_COMPUTE_32F,
                           CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return GRPO_ERR_CUDA;
  }
  return GRPO_OK;
}

// ---- allocation-free forward entry point -----------------------------------------------------
//
// For callers that cannot allocate device memory when they need the loss: a serving or
// scoring process that has handed all device memory to its own pool (KV cache, a caching
// allocator) so that a fresh cudaMalloc would fail or force the pool to shrink, or a code path
// that must not risk the implicit device synchronisation that cudaMalloc / cudaFree can
// cause. Such a caller still passes its inputs and outputs; the forward pass's scratch
// (per-token vocabulary-tile softmax partials, target logits, LSE, coefficients) lives in the
// file-scope array below instead of a caller workspace.
//
// The array is a device symbol: every GPU that loads this library holds its 16 MiB until the
// process exits. In host code its name only stands in for the symbol; the device address is
// looked up once per device (with that device current) by cudaGetSymbolAddress and passed to
// the kernels.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_lmhead_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch array on the current device; the first call on a device does
// the lookup and caches it (the GEMM launcher sets the kernel's shared-memory limit on its own
// first launch on the device).
int noalloc_setup(void** scratch) {
  static void* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return GRPO_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return GRPO_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return GRPO_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *scratch = addr[dev];
  return GRPO_OK;
}

}  // namespace

extern "C" GRPO_API size_t grpo_lmhead_forward_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" GRPO_API int grpo_lmhead_forward_noalloc(const void* h, const void* W, int64_t T, int64_t V,
                                                    int64_t H, const int32_t* target, const float* old_logp,
                                                    const float* adv_tok, const uint8_t* mask, float clip_eps,
                                                    float grad_scale, float* loss_tok, float* logp_tok,
                                                    grpo_step_acc* acc, void* stream) {
  if (T < 0 || V < 1 || H < BK || H % BK != 0 || !acc) return GRPO_ERR_INVALID;
  if (T == 0) return GRPO_OK;
  if (!h || !W || !target || !adv_tok || !mask || !loss_tok) return GRPO_ERR_INVALID;
  if (((uintptr_t)h | (uintptr_t)W) & 15u) return GRPO_ERR_INVALID;
  if (T > INT32_MAX / 2 || V > INT32_MAX / 2) return GRPO_ERR_INVALID;
  // the forward pass uses the workspace layout up to (not including) the dlogits chunk
  const WsLayout ws = ws_layout(T, V, kDefaultVChunk);
  if (ws.dz > kNoAllocScratchBytes) return GRPO_ERR_CAPACITY;
  void* scratch = nullptr;
  const int rc = noalloc_setup(&scratch);
  if (rc != GRPO_OK) return rc;
  uint8_t* wsb = static_cast<uint8_t*>(scratch);
  float* part_m = reinterpret_cast<float*>(wsb + ws.part_m);
  float* part_s = reinterpret_cast<float*>(wsb + ws.part_s);
  float* zy = reinterpret_cast<float*>(wsb + ws.zy);
  float* lse2 = reinterpret_cast<float*>(wsb + ws.lse2);
  float* coef = reinterpret_cast<float*>(wsb + ws.coef);

  const bool pair = use_pair();
  CUtensorMap map_h, map_w;
  if (!make_maps(&map_h, &map_w, h, W, T, V, H, pair)) return GRPO_ERR_UNSUPPORTED;
  const cudaStream_t st = as_stream(stream);
  GemmArgs g{};
  g.T = T;
  g.V = V;
  g.H = H;
  g.n_row_tiles = (int)((T + BM - 1) / BM);
  g.target = target;
  g.part_m = part_m;
  g.part_s = part_s;
  g.zy = zy;
  g.lse2 = lse2;
  g.coef = coef;
  g.acc = acc;
  g.mode = 0;
  g.col_tile0 = 0;
  g.n_col_tiles = ws.n_col_tiles;
  const int lrc = launch_gemm(pair, map_h, map_w, g, st);
  if (lrc != GRPO_OK) return lrc;
  reduce_kernel<<<(unsigned)((T + 255) / 256), 256, 0, st>>>(T, ws.n_col_tiles, part_m, part_s, zy, target, V,
                                                              old_logp, adv_tok, mask, clip_eps, grad_scale, lse2,
                                                              coef, loss_tok, logp_tok, acc);
  GRPO_CUDA_TRY(cudaGetLastError());
  return GRPO_OK;
}
