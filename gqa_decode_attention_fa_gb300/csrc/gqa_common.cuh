// Shared definitions of the decode-attention kernels: geometry constants, the split-KV
// work partition (host and device), kernel parameter blocks and thin inline-PTX wrappers
// for mbarrier, TMA copies, ldmatrix, movmatrix and mma.sync.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gqa_decode.h"

namespace gqa {

constexpr int kHeadDim = 128;
constexpr int kTile = 64;                  // tokens per KV tile = one cache page
constexpr int kHalfRowBytes = 128;         // one half (64 dims) of a bf16 head row
constexpr int kHalfTileBytes = kTile * kHalfRowBytes;   // 8 KiB: 64 rows x 128 B
constexpr int kConsumerWarps = 6;          // warps that run the softmax/mma per CTA
constexpr int kStages = 6;                 // depth of the shared-memory KV ring
// Tile i uses stage i % kStages and consumer warp i % kConsumerWarps.  A consumer waits on
// a stage's "full" barrier by phase parity, which is only unambiguous while the waiter is
// at most one phase ahead of the barrier; tying every stage to a single consumer warp
// (kStages a multiple of kConsumerWarps) guarantees that, because a warp only waits for a
// stage's next fill after it has released the previous one itself.
static_assert(kStages % kConsumerWarps == 0, "each stage must belong to exactly one consumer warp");
constexpr int kThreadsAttn = 32 * (kConsumerWarps + 1);  // + one producer (TMA) warp
constexpr long long kSpinLimitCycles = 4000000000LL;      // ~2 s at 2 GHz

// Split-KV work partition ------------------------------------------------------------
// Tiles are numbered sequence-major, then KV head, then 64-token tile:
//   seg = b * H_kv + kv covers tiles [pre[b] + kv * nt(b), pre[b] + (kv+1) * nt(b)),
//   pre[b] = H_kv * sum_{b' < b} nt(b'),  nt(b) = ceil(L_b / 64).
// Worker w of W owns the contiguous range [T*w/W, T*(w+1)/W) of the T tiles (the
// contiguous-block placement of ADR-0060 section 2.1 applied to the whole batch), and
// consumer warp c of that worker takes local tiles i = c, c + kConsumerWarps, ...  The
// partial of (segment seg, worker w, warp c) lives in slot seg + w, row group
// (seg + w) * kConsumerWarps + c: as one walks the tiles in order, seg + w strictly
// increases from one (segment, worker) piece to the next, so slots never collide and
// B*H_kv + W - 1 slots suffice.

__host__ __device__ inline int tiles_of(int L, int max_seq) {
  return (L >= 1 && L <= max_seq) ? (L + kTile - 1) / kTile : 0;
}
__host__ __device__ inline long long worker_begin(long long T, int W, int w) {
  return (T * (long long)w) / (long long)W;
}
// The worker whose range holds tile x (0 <= x < T).
__host__ __device__ inline int worker_of(long long T, int W, long long x) {
  return (int)(((x + 1) * (long long)W - 1) / T);
}
// Does consumer warp c take any local tile index in [i0, i1)?
__host__ __device__ inline bool warp_has_tile(long long i0, long long i1, int c) {
  long long n = i1 - i0;
  if (n <= 0) return false;
  if (n >= kConsumerWarps) return true;
  long long first = ((c - i0) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
  return first < n;
}

// Kernel parameter blocks -------------------------------------------------------------

struct RopeTableParams {
  float4 *rope_dw;                          // [max_seq][64] (cos_hi, sin_hi, cos_lo, sin_lo)
  float2 *rope_tab32;                       // [max_seq][64] (cos, sin) rounded to binary32
  int max_seq;
  double inv_freq[kHeadDim / 2];            // theta^(-2i/d), i < 64
};

struct AttnParams {
  const int32_t *seq_lens, *page_table, *positions;
  const uint16_t *q_new;                    // [B,Hq,d] new-token queries (rotated by this kernel)
  const uint16_t *k_new, *v_new;            // [B,Hkv,d] new-token rows (appended by this kernel)
  uint16_t *k_cache, *v_cache;              // the caches (the TMA maps view the same memory)
  const uint16_t *q_norm_w, *k_norm_w;      // [d] or null
  const float4 *rope_dw;                    // [max_seq][64] (cos, sin) as double-word hi, lo
  const float2 *rope_tab32;                 // [max_seq][64] (cos, sin) rounded to binary32
  uint16_t *q_rot;                          // [B,Hq,d] copy of the rotated bf16 queries
  int inputs_in_host_memory;                // q/k/v_new, seq_lens, positions are mapped host memory
  int2 *spec;                               // [W][kStages] (cache row, KV head) of each worker's
                                            // first tiles at the previous launch (row < 0: none),
                                            // or null
  float *part_o;                            // [slots * kConsumerWarps * G][128]
  float *part_ml;                           // [slots * kConsumerWarps * G][2]  (m in log2 units, l)
  uint32_t *err;
  uint16_t *out;                            // [B,Hq,d]: written by the single-launch form only
  int B, Hq, Hkv, G;
  int paged, max_seq, max_blocks, num_blocks;
  int csize;                                // single-launch form: CTAs per segment (cluster size)
  int spec_tiles;                           // single-launch form: tiles of the longest segment the
                                            // plan expects (its first tiles are loaded before the
                                            // length is read)
  const int32_t *seg_order;                 // single-launch form: cluster i streams segment
                                            // seg_order[i] (b H_kv + kv), or i when null
  double eps;
  float scale_log2;                         // log2(e) / sqrt(d)
};

struct CombineParams {
  const int32_t *seq_lens;
  const float *part_o, *part_ml;
  uint16_t *out;                            // [B,Hq,d]
  int B, Hq, Hkv, G, W, max_seq;
};

// Inline PTX -----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory buffer advanced to a 1024-byte boundary (the period of the
// 128-byte TMA swizzle) by pointer arithmetic on the buffer itself, so that the compiler
// still sees the result as shared memory and emits shared-memory loads and stores for it
// (an integer round trip would leave it a generic pointer).
__device__ __forceinline__ uint8_t *align_smem_1024(uint8_t *raw) {
  return raw + ((1024u - (smem_addr(raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete; gives up after
// kSpinLimitCycles and returns false (the caller records GQA_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kSpinLimitCycles) return false;
  }
  return true;
}

// Programmatic dependent launch: every kernel of the step is launched so that it may
// start while the previous kernel in the stream drains; each one waits here before it
// touches memory an earlier kernel writes, and then lets the next kernel launch.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters: every thread of every CTA of the cluster arrives (release) and
// later waits (acquire); the wait returns once all of them have arrived.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// An arrive that orders nothing (no release): for a barrier whose only job is to keep
// CTAs alive until every one of them has observed its own receptions complete.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
// Stores into another CTA's shared memory (a shared::cluster address) that count their
// bytes on that CTA's mbarrier (also a shared::cluster address), from registers.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_v2f32(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 3-D tiled TMA load global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// TMA prefetch of a 3-D tile into L2 (no shared memory, no barrier); out-of-range
// coordinates are allowed, as for loads.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
// Bulk copy global -> this CTA's shared memory of `bytes` (both addresses 16-byte aligned,
// a multiple of 16 bytes), completion counted on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two floats -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float bf16_lo_to_float(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_to_float(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Byte offset of (row, 16-byte chunk) in a [rows][128 B] buffer written by a TMA box with
// 128-byte swizzling: chunk index XOR (row mod 8).  The buffer must be 1024-byte aligned.
__host__ __device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace gqa
