// Grouped expert GEMMs for bf16 layers on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// Pages: "MoE Architecture" (vanos001.github.io) "Efficient Batched MoE" (one
// grouped computation over the experts instead of a per-expert loop),
// SwiGLUExpert / StandardExpert, HybridMoE (shared expert on every token);
// "Mixture of Experts" (aigrafen.se) MoE code (out[index] += w * expert(x));
// "Mixture of Experts (MoE)" (learn.starphix.com) "Shared + Specialized".
//
// One launch computes every tile of two families of groups:
//   up-projection   family 0: expert e's rows of xp  x  W1[e] (+W3[e])  -> H
//                   family 1: all tokens of x  x  Ws1[s] (+Ws3[s])      -> Hs[:, s*Fs...]
//   down-projection family 0: expert e's rows of H   x  W2[e]           -> Yp (x row gate)
//                   family 1: all tokens of Hs x [Ws2[0] | Ws2[1] | ...] -> Ys fp32 (the shared
//                             experts concatenated along K, so their sum comes out of one
//                             accumulator)
// A group's rows come from the device-side expert offsets, so no host sync is
// needed; every CTA builds the same tile prefix over the groups and walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... (persistent, one CTA per SM); a last wave
// that would keep at most half the CTAs busy is cut into half-width tiles instead.
//
// Tile 128 x BN x 64, K-major operands in 128-byte-swizzled shared memory.
// Warp roles: warp 0 issues TMA loads into a STAGES-deep ring, warp 1 issues
// tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM accumulators, warps 2-13
// drain the other accumulator with tcgen05.ld (warp w reads TMEM lanes
// 32*(w%4)...), apply the epilogue (GELU + bias, SiLU x gate, or bias x row gate;
// two columns per packed fp32x2 operation), and store through TMA. SwiGLU tiles
// load BN/2 rows of W1 and BN/2 rows of W3 into one BN-row B tile, so one MMA
// fills both halves of the accumulator.
//
// Pair form (down-projection of large batches): clusters of two CTAs compute
// 256 x BN tiles with the M = 256 tcgen05.mma of a CTA pair. Each CTA stages its own
// 128 rows of A and half of B; both halves' copies complete on the leader's
// barrier, the leader issues the MMAs, its commits arrive at both CTAs, and each CTA
// drains its own 128 accumulator rows, the peer signalling the leader when done.
//
// MXFP8 form (layers whose routed experts compute in MXFP8, "Mixture of Experts (MoE)"
// (learn.starphix.com), "Quantization"): A and B are E4M3 codes with an E8M0 scale per
// 32 elements along K, multiplied by tcgen05.mma kind::mxf8f6f4 with block scaling
// (M=128, N=128, K=32 per instruction, 128 codes per stage). The producer warp's lanes
// copy each stage's scale bytes into shared memory (cp.async), the MMA thread moves
// them into tensor memory (tcgen05.cp) ahead of the stage's MMAs, and the
// up-projection's epilogue quantises H to MXFP8 for the down-projection.
//
// Every mbarrier wait is bounded by the global timer; on expiry the CTA records
// MOE_ERR_TIMEOUT in the workspace error word, waits (bounded) for its own TMA
// copies and MMAs in flight, frees its TMEM and exits.
#include <cuda.h>

#include <cstdlib>

#include "act.cuh"
#include "common.cuh"
#include "internal.h"
#include "mx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 12;  // 3 per TMEM lane quadrant (warps sharing a quadrant split its 32-column chunks)
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kMaxGroups = 512 + 64;  // E <= 512 routed + S <= 64 shared groups
constexpr unsigned long long kTimeoutNs = 2000000000ull;

enum Epi { kGelu = 0, kSwiglu = 1, kLinear = 2, kLogits = 3 };

struct Family {
  int32_t groups;       // groups in the family (0 = unused)
  int32_t m_from_off;   // 1: group g has rows [off[g], off[g+1]); 0: rows [0, m_fixed)
  int32_t m_fixed;
  int32_t n_tiles;      // output column tiles per group
  int32_t k_blocks;     // K / BK
  int32_t kseg_blocks;  // B is cut along K into segments of this many blocks
  int32_t b_rows_group; // B-map row offset of group g: g * b_rows_group
  int32_t b_rows_kseg;  // B-map row offset of K segment s: s * b_rows_kseg
  int32_t a_map, b_map, b3_map;
  int32_t k_group;      // K-block offset of group g: g * k_group (split-K groups), else 0
  void* out;
  int64_t ld_out;         // elements between output rows
  int64_t out_col_group;  // output column offset of group g: g * out_col_group
  const __nv_bfloat16* bias;
  int64_t bias_group;       // bias offset of group g
  int64_t bias_sum_stride;  // stride between summed bias vectors
  int32_t bias_nsum;        // bias vectors summed per column (0 = no bias)
  int32_t pad1;
  const float* row_gate;  // per output row scale, or null
  const float* bias_f32;  // kLogits: fp32 per-column bias, or null
  int64_t n_valid;        // kLogits: columns < n_valid are stored
  int32_t tma_out;        // bf16 outputs: store full 32-row blocks through the family's output tensor map
  int32_t gather_n;       // gather_rows: rows of the gathered matrix (bounds of the row ids)
  const int32_t* gather_rows;  // non-null: A row r of a group is row gather_rows[r] of the a_map matrix,
                               // loaded with tile::gather4 (a_map has one-row boxes)
  // MXFP8 form: A and B are E4M3 codes (the maps' rows are bytes) with one E8M0 scale
  // byte per 32 codes along K, scales row-major [rows, K / 32]; H tiles are stored as
  // codes + scales (out_scale) for the next GEMM.
  int32_t a_rows;           // rows of the A matrix (bound of the A scale reads)
  const uint8_t* a_scale;   // [a_rows, a_scale_ld]
  int64_t a_scale_ld;
  const uint8_t* b_scale;   // rows of b_map
  const uint8_t* b3_scale;  // rows of b3_map
  int64_t scale_ld;
  uint8_t* out_scale;       // [rows of out, out_scale_ld]
  int64_t out_scale_ld;
};

struct Params {
  Family fam[2];
  const int32_t* expert_off;
  int32_t* status;
  unsigned long long wait_ns;  // bound on each pipeline wait (teardown drains keep kTimeoutNs)
};

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Test for completion of the phase with the given parity. kSleep: a waiting
// thread is suspended in hardware (up to ~1 ms) until the phase completes, so a
// long wait costs no issue slots (epilogue warps waiting for a whole mainloop);
// otherwise the test returns at once (the single producer and MMA threads, whose
// short waits are on the critical path, poll).
template <bool kSleep>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if (kSleep) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
  } else {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}
// Bounded wait: false after limit_ns or once another role has aborted.
template <bool kSleep>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait<kSleep>(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < (kSleep ? 1 : 64); ++i)
      if (mbar_try_wait<kSleep>(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Four rows of a 2-D tensor map with one-row boxes (rows r0..r3, columns x .. x + box - 1)
// into four consecutive box rows of shared memory at dst (completion counted on bar).
// The 128-byte swizzle follows the shared-memory address, so four groups of rows
// written at 512-byte steps land exactly as one 128-row box would.
__device__ __forceinline__ void tma_gather4(const CUtensorMap* map, uint64_t* bar, void* dst, int32_t x, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}
// Bulk tensor store smem -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until no committed bulk store is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on bar once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- CTA-pair forms (cluster of 2; the even CTA is the leader that issues the MMAs) ----
// Tensor memory is allocated and freed collectively by one warp of each CTA of the
// pair; an M = 256 MMA takes rows 0-127 of A from the leader's shared memory and
// rows 128-255 from the peer's, B's first N/2 rows from the leader and the rest from
// the peer (same shared-memory offsets in both), and writes accumulator rows 0-127
// to the leader's tensor memory, rows 128-255 to the peer's.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on the
// leader's mbarrier (`bar_cluster`: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar_cluster, void* dst, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the mbarrier at this offset in both CTAs of the pair once the MMAs
// issued so far have completed
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_alloc_t(uint32_t* dst_smem, uint32_t ncols) {
  if constexpr (PAIR) tmem_alloc_pair(dst_smem, ncols); else tmem_alloc(dst_smem, ncols);
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc_t(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR) tmem_dealloc_pair(taddr, ncols); else tmem_dealloc(taddr, ncols);
}
template <bool PAIR>
__device__ __forceinline__ void umma_commit_t(uint64_t* bar) {
  if constexpr (PAIR) umma_commit_pair(bar); else umma_commit(bar);
}
// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Waits for this thread's tcgen05.ld results; the registers are in/out operands so
// no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// Orders the registers r after an earlier wait without waiting again.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row core groups 1024 bytes apart (SBO),
// LBO unused for swizzled K-major (set to 1), descriptor version 1, layout 2 =
// SWIZZLE_128B. Advancing K by 16 bf16 inside the atom adds 32 bytes to the start.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  desc |= (uint64_t)1 << 16;
  desc |= (uint64_t)(1024 >> 4) << 32;
  desc |= (uint64_t)1 << 46;
  desc |= (uint64_t)2 << 61;
  return desc;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A and B E4M3 (format 0),
// both K-major, scale factors E8M0 (bit 23), M x N; the scale-factor IDs (bits 29-30
// for A, 4-5 for B) pick the byte of each 32-bit tensor-memory scale word, i.e. which
// 32-element K block of the stage the MMA uses.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 23) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}
// D (+)= (A x 2^sA) (B x 2^sB)^T over K = 32 E4M3 elements, scales read from tensor memory.
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.block32 [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :
      : "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Shared-memory descriptor of a 32-row x 16-byte scale atom (no swizzle: 8-row core
// matrices of 128 contiguous bytes, 128 bytes apart), the source of tcgen05.cp.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  desc |= (uint64_t)(128 >> 4) << 16;
  desc |= (uint64_t)(128 >> 4) << 32;
  desc |= (uint64_t)1 << 46;
  return desc;
}
// Copy a scale atom (32 rows of 16 bytes) into 4 tensor-memory columns of every lane
// quadrant: lane 32q + i, column c holds the 4 scale bytes of row 32c + i. The MMA
// reads row r's scale at lane r % 32 (+ 32q), column r / 32, byte = scale-factor ID.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// 4-byte asynchronous copy global -> shared; src_bytes 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool read) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(read ? 4 : 0)
               : "memory");
}
// The barrier receives one arrival once all of this thread's earlier cp.async copies
// have landed (counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// PAIR: the tile is 256 x BN on a CTA pair; each CTA stages its 128 rows of A and
// half (BN / 2 rows) of B.
// MXR > 0, the MXFP8 form (tcgen05 kind::mxf8f6f4 with E8M0 block scales): A and B
// arrive as E4M3 codes in 128-byte K atoms (128 codes of a row, one swizzle atom, as
// 64 bf16 are), and each stage's scale bytes go to a third ring of 32 x 16-byte atoms
// that tcgen05.cp moves into tensor memory beside the accumulators. A tile covers MXR
// rows of A. MXR = 32 (decode batches: the weight stream is the work) takes two K atoms
// per stage, 32 KB of weights, since a stage's fixed costs (barriers, scale copies)
// otherwise bound the stream (measured: 16 KB stages stream at about half the HBM
// rate of 32 KB ones); its A atoms are 4 KB boxes, and the M = 128 MMA reads the 16 KB
// after an atom's start, whose extra rows are never stored.
constexpr int mx_atoms(int mxr) { return mxr == 32 ? 2 : 1; }

// kStaging: the epilogue stores through TMA and needs its per-warp staging blocks (every
// form but the MXFP8 up-projection, whose epilogue writes codes and scales with plain
// stores and gives that shared memory to the operand ring instead).
template <int BN, bool PAIR = false, int MXR = 0, bool kStaging = true>
struct Cfg {
  static constexpr bool kMx = MXR != 0;
  static constexpr int kTileRows = kMx ? MXR : BM;  // A rows of a tile
  static constexpr int kAtoms = kMx ? mx_atoms(MXR) : 1;  // 128-byte K atoms per stage
  static constexpr int kStageK = kMx ? 128 * kAtoms : BK;  // K elements per stage
  static constexpr int kStagingBytes = 2048;               // per epilogue warp: 32 rows x 64 B
  static constexpr int kAAtomBytes = kTileRows * 128;
  static constexpr int kBAtomBytes = (PAIR ? BN / 2 : BN) * 128;
  static constexpr int kABytes = kAtoms * kAAtomBytes;
  static constexpr int kBBytes = kAtoms * kBAtomBytes;
  static constexpr int kSFAtomBytes = kMx ? 512 * (1 + BN / 128) : 0;  // per K atom: A's scale atom, then B's
  static constexpr int kSFBytes = kAtoms * kSFAtomBytes;
  static constexpr int kTxBytes = kABytes + kBBytes;  // TMA bytes per stage
  static constexpr int kStageBytes = kTxBytes + kSFBytes;
  static constexpr int kStagingTotal = kStaging ? kEpiWarps * kStagingBytes : 0;
  static constexpr int kRingBudget = 192 * 1024 + (kEpiWarps * kStagingBytes - kStagingTotal);
  static constexpr int kStages = kRingBudget / kStageBytes > 8 ? 8 : kRingBudget / kStageBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;  // A slots, B slots, scale atoms
  static constexpr int kSFAtomCols = 4 + 4 * (BN / 128);     // tensor-memory columns of one K atom's scales
  static constexpr int kSFCols = kAtoms * kSFAtomCols;
  static constexpr int kTmemCols = kMx ? 512 : 2 * BN;  // two accumulators (+ the scale ring)
  static constexpr size_t kSmem = (size_t)kRingBytes + (size_t)kStagingTotal + 1024;
  static_assert(!kMx || (!PAIR && BN == 128), "MXFP8 tiles: single CTAs, 128 columns");
  static_assert(!kMx || 2 * BN + kStages * kSFCols <= 512, "accumulators and scales fit tensor memory");
  static_assert(kStages >= 3, "pipeline depth");
  // the M = 128 MMA reads 16 KB of A from an atom's start: past a short atom come later
  // atoms and slots, then the B slots and the scale atoms, all shared memory of this block
  static_assert((kStages - 1) * kABytes + (kAtoms - 1) * kAAtomBytes + BM * 128 <= kRingBytes, "A overhang");
};

struct TileInfo {
  int fam, g, mt, nt, m, a_row0;
};

// The work of one CTA (or CTA pair): tiles b, b + W, b + 2W, ... When `split`, the
// last wave's tiles (fewer than half the CTAs) are cut instead into two halves of
// BN / 2 output columns, half h of tile nwave * W + j going to CTA 2j + h, so the
// last wave ends after about half a tile's time.
struct Walk {
  int b, W, total, nwave, split;
  __device__ __forceinline__ bool item(int it, int& tile, int& half) const {
    half = -1;
    if (!split || it < nwave) {
      tile = b + it * W;
      return tile < total;
    }
    if (it == nwave && b < 2 * (total - nwave * W)) {
      tile = nwave * W + (b >> 1);
      half = b & 1;
      return true;
    }
    return false;
  }
};

// Tile `tile` of the prefix s_start. PAIR: tiles are 256-row pair tiles and the CTA
// of rank `half` in the pair takes their 128-row half `half`.
template <bool PAIR = false, int TR = BM>
__device__ __forceinline__ TileInfo decode_tile(int tile, const int32_t* s_start, int G, int G0,
                                                const Family* fams, const int32_t* off, int half = 0) {
  int lo = 0, hi = G;  // last group whose start <= tile
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] <= tile) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.fam = lo < G0 ? 0 : 1;
  ti.g = lo < G0 ? lo : lo - G0;
  const Family& F = fams[ti.fam];
  int row0;
  if (F.m_from_off) {
    row0 = off[ti.g];
    ti.m = off[ti.g + 1] - row0;
  } else {
    row0 = 0;
    ti.m = F.m_fixed;
  }
  const int m_tiles = PAIR ? (ti.m + 2 * BM - 1) / (2 * BM) : (ti.m + TR - 1) / TR;
  const int local = tile - s_start[lo];
  ti.nt = local / m_tiles;
  ti.mt = local - ti.nt * m_tiles;
  if (PAIR) ti.mt = 2 * ti.mt + half;
  ti.a_row0 = row0 + ti.mt * TR;
  return ti;
}

__device__ __forceinline__ const CUtensorMap* pick_map(int i, const CUtensorMap& m0, const CUtensorMap& m1,
                                                       const CUtensorMap& m2, const CUtensorMap& m3,
                                                       const CUtensorMap& m4, const CUtensorMap& m5) {
  switch (i) {
    case 0: return &m0;
    case 1: return &m1;
    case 2: return &m2;
    case 3: return &m3;
    case 4: return &m4;
    default: return &m5;
  }
}

template <int BN, int EPI, bool PAIR, int MXR = 0>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap m0, const __grid_constant__ CUtensorMap m1,
                        const __grid_constant__ CUtensorMap m2, const __grid_constant__ CUtensorMap m3,
                        const __grid_constant__ CUtensorMap m4, const __grid_constant__ CUtensorMap m5,
                        const __grid_constant__ CUtensorMap o0, const __grid_constant__ CUtensorMap o1,
                        const __grid_constant__ Params P) {

  using C = Cfg<BN, PAIR, MXR, !(MXR != 0 && EPI != kLinear)>;
  constexpr bool kMx = C::kMx;
  constexpr int kTR = C::kTileRows;
  constexpr int kKE = C::kStageK;
  constexpr int kStages = C::kStages;
  constexpr int kOutCols = EPI == kSwiglu ? BN / 2 : BN;
  constexpr uint32_t kIdesc = idesc_bf16(PAIR ? 2 * BM : BM, BN);
  // half tiles for the last wave (bf16 single CTAs): N = BN / 2 against half of the staged B
  // tile (GELU, linear), or two N = BN / 4 MMAs against a quarter of each of its W1 and W3
  // halves (SwiGLU)
  // (SwiGLU halves: output columns [h BN/4, (h + 1) BN/4), from W1 and W3 rows of that range,
  // whole 32-column chunks, so BN >= 128)
  constexpr bool kCanSplit = !PAIR && !kMx && (EPI == kGelu || EPI == kLinear || (EPI == kSwiglu && BN >= 128));
  // MXFP8 decode tiles (32 A rows): warp 2, whose TMEM lane quadrant holds no rows of
  // such a tile, copies the scale bytes, so the TMA producer only issues tensor copies
  constexpr bool kScaleWarp = kMx && kTR == 32;
  constexpr int kDrainWarps = kEpiWarps - (kScaleWarp ? 1 : 0);
  constexpr uint32_t kIdescHalf = idesc_bf16(BM, BN / 2);
  constexpr uint32_t kIdescQuarter = idesc_bf16(BM, BN / 4);

  extern __shared__ uint8_t smem_raw[];
  // full_bar: a stage's operands have landed (MXFP8 form: and the 32 producer lanes'
  // scale copies); empty_bar: the MMAs are done with the stage.
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], done_bar;
  __shared__ uint32_t s_tmem_base;
  __shared__ int32_t s_start[kMaxGroups + 1];
  __shared__ Family s_fam[2];
  __shared__ int32_t s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // PAIR: rank 0 (leader) issues the MMAs and owns the full / accumulator-empty barriers
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int walk0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int walk_step = PAIR ? (int)nclusters_x() : (int)gridDim.x;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * C::kABytes;
  uint8_t* sSF = sB + kStages * C::kBBytes;  // MXFP8 form: the scale atoms of each stage
  const int32_t* off = P.expert_off;

  if (threadIdx.x == 0) {
    s_fam[0] = P.fam[0];
    s_fam[1] = P.fam[1];
    s_abort = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], kMx ? 33 : 1);  // MXFP8: + one cp.async arrival per producer lane
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], PAIR ? 2 * kEpiWarps : kDrainWarps);
    }
    mbar_init(&done_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Set-up that reads nothing earlier kernels wrote runs before the dependency wait, so
  // it overlaps the previous kernel's tail: the tensor-map prefetch and the TMEM
  // allocation (a previous CTA of this kernel cannot share the SM: its shared memory
  // takes the SM's whole budget; the other kernels of the forward use no TMEM).
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&m0);
    prefetch_tensormap(&m1);
    prefetch_tensormap(&m2);
    prefetch_tensormap(&m3);
    prefetch_tensormap(&m4);
    prefetch_tensormap(&m5);
    prefetch_tensormap(&o0);
    prefetch_tensormap(&o1);
  }
  if (warp == 1) tmem_alloc_t<PAIR>(&s_tmem_base, C::kTmemCols);
  pdl_wait();  // expert offsets, operands: written by the previous kernels of the stream
  pdl_launch_next();
  // tile prefix over all groups of both families (same in every CTA)
  const int G0 = P.fam[0].groups, G = G0 + P.fam[1].groups;
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int tiles = 0;
      if (g < G) {
        const Family& F = g < G0 ? P.fam[0] : P.fam[1];
        const int gl = g < G0 ? g : g - G0;
        const int m = F.m_from_off ? off[gl + 1] - off[gl] : F.m_fixed;
        tiles = (PAIR ? (m + 2 * BM - 1) / (2 * BM) : (m + kTR - 1) / kTR) * F.n_tiles;
      }
      const int inc = warp_inclusive_scan(tiles);
      if (g < G) s_start[g] = carry + inc - tiles;
      carry += __shfl_sync(kFull, inc, 31);
    }
    if (lane == 0) s_start[G] = carry;
  }
  tc_fence_before();
  __syncthreads();
  // PAIR: both CTAs' barriers are initialised before either CTA signals the other's
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = s_start[G];
  Walk walk;
  walk.b = walk0;
  walk.W = walk_step;
  walk.total = total;
  walk.nwave = total / walk_step;
  walk.split = kCanSplit && total % walk_step != 0 && 2 * (total % walk_step) <= walk_step;
  int first_tile, first_half;
  if (!walk.item(0, first_tile, first_half)) {  // uniform across the CTA (and the pair): nothing to do
    if (warp == 1) tmem_dealloc_t<PAIR>(tmem_base, C::kTmemCols);
    return;
  }
  volatile int32_t* abort_flag = &s_abort;
  // MXFP8 form: the 32 lanes of the calling warp copy stage `stage`'s scale bytes (4 per
  // row and K atom: its four 32-element blocks) into the tensor-memory copy layout, row r
  // of a 128-row atom at byte 16 (r % 32) + 4 (r / 32), then each lane adds one arrival
  // on the stage's barrier once its copies have landed.
  auto mx_scale_copies = [&](const TileInfo& ti, const Family& F, int kb, int stage) {
#pragma unroll
    for (int a = 0; a < C::kAtoms; ++a) {
      uint8_t* sf = sSF + stage * C::kSFBytes + a * C::kSFAtomBytes;
      const int sc = 4 * (kb * C::kAtoms + a);  // the atom's 4 scale bytes in a row's scales
#pragma unroll
      for (int j = 0; j < kTR / 32; ++j) {  // A rows past the matrix read nothing (zeros)
        const int row = ti.a_row0 + lane + 32 * j;
        const bool in = row < F.a_rows;
        cp_async4(sf + 16 * lane + 4 * j, F.a_scale + (int64_t)(in ? row : 0) * F.a_scale_ld + sc, in);
      }
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) {  // B rows: W1 then W3 halves (SwiGLU), else BN rows
        const int n = lane + 32 * j;
        const uint8_t* src;
        if (EPI == kSwiglu) {
          const bool up = n >= BN / 2;
          const int64_t brow =
              (int64_t)ti.g * F.b_rows_group + (int64_t)ti.nt * (BN / 2) + (up ? n - BN / 2 : n);
          src = (up ? F.b3_scale : F.b_scale) + brow * F.scale_ld;
        } else {
          src = F.b_scale + ((int64_t)ti.g * F.b_rows_group + (int64_t)ti.nt * BN + n) * F.scale_ld;
        }
        cp_async4(sf + 512 * (1 + (j >> 2)) + 16 * lane + 4 * (j & 3), src + sc, true);
      }
    }
    cp_async_arrive_noinc(&full_bar[stage]);
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // Lane 0 waits for free stages and issues the copies; for a gathering family the
    // 32 lanes issue one tile::gather4 each (4 of the tile's 128 A rows, row ids held in
    // registers for the tile), after lane 0 has set the stage's expected bytes. MXFP8
    // form: the 32 lanes also copy the stage's scale bytes (mx_scale_copies), or the
    // scale warp does (decode tiles).
    int stage = 0;
    uint32_t phase = 0;
    int32_t last_parity[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) last_parity[s] = -1;
    bool ok = true;
    for (int it = 0, tile, half; ok && walk.item(it, tile, half); ++it) {
      const TileInfo ti = decode_tile<PAIR, kTR>(tile, s_start, G, G0, s_fam, off, (int)rank);
      const Family& F = s_fam[ti.fam];
      const CUtensorMap* ma = pick_map(F.a_map, m0, m1, m2, m3, m4, m5);
      const CUtensorMap* mb = pick_map(F.b_map, m0, m1, m2, m3, m4, m5);
      const CUtensorMap* mb3 = pick_map(F.b3_map, m0, m1, m2, m3, m4, m5);
      const int k0 = ti.g * F.k_group;  // split-K groups start further along K
      const bool gather = !PAIR && F.gather_rows != nullptr;
      int32_t gr[4] = {0, 0, 0, 0};
      if (gather) {
        // rows past the group's end repeat its first row (their results are not stored)
        const int row0 = ti.a_row0 - ti.mt * BM;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane * 4 + i;
          const int src = ti.mt * BM + r < ti.m ? ti.a_row0 + r : row0;
          int32_t id = F.gather_rows[src];
          if (id < 0 || id >= F.gather_n) {
            record_error(P.status, kErrIndex, 204, src, id);
            id = 0;
          }
          gr[i] = id;
        }
      }
      for (int kb = 0; kb < F.k_blocks; ++kb) {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait<false>(&empty_bar[stage], phase ^ 1u, abort_flag, P.wait_ns) ? 1 : 0;
        if (!__shfl_sync(kFull, w_ok, 0)) {
          ok = false;
          break;
        }
        const int kseg = kb / F.kseg_blocks;
        const int kin = k0 + kb - kseg * F.kseg_blocks;
        if (lane == 0) {
          if (PAIR) {
            // both CTAs' copies complete on the leader's full barrier, which expects
            // the bytes of the two halves; B: the leader stages rows [0, BN/2) of the
            // tile, the peer rows [BN/2, BN)
            const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0u);
            if (rank == 0) {
              mbar_arrive_expect_tx(&full_bar[stage], 2 * C::kStageBytes);
              last_parity[stage] = (int32_t)phase;
            }
            tma_load_2d_pair(ma, fb, sA + stage * C::kABytes, (k0 + kb) * BK, ti.a_row0);
            if (EPI == kSwiglu) {  // the leader stages the tile's W1 rows, the peer its W3 rows
              const int by = ti.g * F.b_rows_group + kseg * F.b_rows_kseg + ti.nt * (BN / 2);
              tma_load_2d_pair(rank == 0 ? mb : mb3, fb, sB + stage * C::kBBytes, kin * BK, by);
            } else {
              const int by = ti.g * F.b_rows_group + kseg * F.b_rows_kseg + ti.nt * BN + (int)rank * (BN / 2);
              tma_load_2d_pair(mb, fb, sB + stage * C::kBBytes, kin * BK, by);
            }
          } else {
            // a half tile stages the whole B tile too (one BN-row copy: two half-height
            // copies per stage measured slower than the bytes they save)
            mbar_arrive_expect_tx(&full_bar[stage], C::kTxBytes);
            last_parity[stage] = (int32_t)phase;
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a) {  // K atom a of the stage (MXFP8: codes [kKE kb + 128 a, + 128))
              const int ka = (k0 + kb) * kKE + 128 * a, kba = kin * kKE + 128 * a;
              uint8_t* a_dst = sA + stage * C::kABytes + a * C::kAAtomBytes;
              uint8_t* b_dst = sB + stage * C::kBBytes + a * C::kBAtomBytes;
              if (!gather) tma_load_2d(ma, &full_bar[stage], a_dst, ka, ti.a_row0);
              if (EPI == kSwiglu) {
                const int by = ti.g * F.b_rows_group + kseg * F.b_rows_kseg + ti.nt * (BN / 2);
                tma_load_2d(mb, &full_bar[stage], b_dst, kba, by);
                tma_load_2d(mb3, &full_bar[stage], b_dst + (BN / 2) * 128, kba, by);
              } else {
                const int by = ti.g * F.b_rows_group + kseg * F.b_rows_kseg + ti.nt * BN;
                tma_load_2d(mb, &full_bar[stage], b_dst, kba, by);
              }
            }
          }
        }
        if constexpr (kMx && !kScaleWarp) mx_scale_copies(ti, s_fam[ti.fam], kb, stage);
        if (gather) {
          __syncwarp();  // the stage's expected bytes are set before any gathered row lands
          tma_gather4(ma, &full_bar[stage], sA + stage * C::kABytes + lane * (4 * BK * 2), (k0 + kb) * BK, gr[0],
                      gr[1], gr[2], gr[3]);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      record_error(P.status, kErrTimeout, 201, (int32_t)blockIdx.x, 0);
      s_abort = 1;
      // let our own copies land before the CTA's shared memory goes away (every lane's
      // gathers of a stage complete on the same barrier as lane 0's copies). One 2 s
      // bound for all stages: a stage whose scale copies the aborted scale warp never
      // issued does not complete, and by then the tensor copies have long landed.
      const unsigned long long t0 = globaltimer();
      for (int s = 0; s < kStages; ++s)
        if (last_parity[s] >= 0) {
          while (!mbar_try_wait<true>(&full_bar[s], (uint32_t)last_parity[s]) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int it = 0, tile, half; ok && (!PAIR || rank == 0) && walk.item(it, tile, half); ++it) {
        const TileInfo ti = decode_tile<PAIR, kTR>(tile, s_start, G, G0, s_fam, off, (int)rank);
        const int kblocks = s_fam[ti.fam].k_blocks;
        // a half tile multiplies by B's rows [half * BN/2, (half + 1) * BN/2) into accumulator columns [0, BN/2)
        const uint32_t idesc = half < 0 ? kIdesc : kIdescHalf;
        // (SwiGLU: B rows [h BN/4, (h + 1) BN/4) of W1 and the same of W3, BN/2 rows further, into
        // accumulator columns [0, BN/4) and [BN/4, BN/2))
        const uint32_t b_off =
            half < 0 ? 0u : (uint32_t)half * (EPI == kSwiglu ? BN / 4 : BN / 2) * 128;
        if (!mbar_wait<false>(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, P.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait<false>(&full_bar[stage], phase, abort_flag, P.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * C::kABytes);
          const uint32_t b_addr = smem_u32(sB + stage * C::kBBytes) + b_off;
          if constexpr (kMx) {
            // the stage's scale atoms (written through the generic proxy by cp.async) into
            // its tensor-memory columns; a stage's columns are reused only after the stage
            // has been refilled, i.e. after the MMAs that read them have completed
            fence_proxy_async_smem();
#pragma unroll
            for (int a = 0; a < C::kAtoms; ++a) {
              const uint32_t sfa = tmem_base + (uint32_t)(2 * BN + stage * C::kSFCols + a * C::kSFAtomCols);
              const uint32_t sf_smem = smem_u32(sSF + stage * C::kSFBytes + a * C::kSFAtomBytes);
              tc_cp_sf(sfa, sf_desc(sf_smem));
              tc_cp_sf(sfa + 4, sf_desc(sf_smem + 512));
              const uint32_t aa = a_addr + a * C::kAAtomBytes, ba = b_addr + a * C::kBAtomBytes;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K = 32 codes per MMA: the scale word's byte kk
                umma_mx(d_tmem, sw128_desc(aa + kk * 32), sw128_desc(ba + kk * 32), idesc_mx(BM, BN, (uint32_t)kk),
                        sfa, sfa + 4, (kb | a | kk) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              if constexpr (PAIR) {
                umma_bf16_pair(d_tmem, sw128_desc(a_addr + kk * UMMA_K * 2), sw128_desc(b_addr + kk * UMMA_K * 2),
                               kIdesc, (kb | kk) != 0 ? 1u : 0u);
              } else if (EPI == kSwiglu && half >= 0) {
                umma_bf16(d_tmem, sw128_desc(a_addr + kk * UMMA_K * 2), sw128_desc(b_addr + kk * UMMA_K * 2),
                          kIdescQuarter, (kb | kk) != 0 ? 1u : 0u);
                umma_bf16(d_tmem + BN / 4, sw128_desc(a_addr + kk * UMMA_K * 2),
                          sw128_desc(b_addr + (BN / 2) * 128 + kk * UMMA_K * 2), kIdescQuarter, (kb | kk) != 0 ? 1u : 0u);
              } else {
                umma_bf16(d_tmem, sw128_desc(a_addr + kk * UMMA_K * 2), sw128_desc(b_addr + kk * UMMA_K * 2),
                          idesc, (kb | kk) != 0 ? 1u : 0u);
              }
            }
          }
          umma_commit_t<PAIR>(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_t<PAIR>(&tfull_bar[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        record_error(P.status, kErrTimeout, 202, (int32_t)blockIdx.x, 0);
        s_abort = 1;
      }
      // every MMA this thread issued has finished before TMEM is released (PAIR: the
      // leader's commit also tells the peer, whose shared and tensor memory they use)
      if (!PAIR || rank == 0) umma_commit_t<PAIR>(&done_bar);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait<true>(&done_bar, 0u) && globaltimer() - t0 < kTimeoutNs) {
      }
    }
  } else if (kScaleWarp && warp == 2) {
    // ---------------- scale copies (MXFP8 decode tiles) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = 0, tile, half; ok && walk.item(it, tile, half); ++it) {
      const TileInfo ti = decode_tile<false, kTR>(tile, s_start, G, G0, s_fam, off, 0);
      const Family& F = s_fam[ti.fam];
      for (int kb = 0; kb < F.k_blocks; ++kb) {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait<false>(&empty_bar[stage], phase ^ 1u, abort_flag, P.wait_ns) ? 1 : 0;
        if (!__shfl_sync(kFull, w_ok, 0)) {
          ok = false;
          break;
        }
        mx_scale_copies(ti, F, kb, stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (!ok && lane == 0) {
      record_error(P.status, kErrTimeout, 205, (int32_t)blockIdx.x, 0);
      s_abort = 1;
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int ew = warp - 2;
    const int q = warp & 3;       // TMEM lane quadrant this warp may read
    const int part = ew >> 2;     // which interleaved share of the 32-column chunks
    const int r = q * 32 + lane;  // row inside the tile
    uint8_t* staging = smem + C::kRingBytes + (C::kStagingTotal ? ew * C::kStagingBytes : 0);  // (TMA stores only)
    bool store_pending = false;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0, tile, half; walk.item(it, tile, half); ++it) {
      const TileInfo ti = decode_tile<PAIR, kTR>(tile, s_start, G, G0, s_fam, off, (int)rank);
      const Family& F = s_fam[ti.fam];
      // output columns of this CTA's share of the tile: all, or one half (accumulator columns 0..)
      constexpr int kHalfCols = EPI == kSwiglu ? BN / 4 : BN / 2;
      const int out_cols = half < 0 ? kOutCols : kHalfCols;
      const int col_shift = half < 0 ? 0 : half * kHalfCols;
      const int u_cols = half < 0 ? BN / 2 : BN / 4;  // SwiGLU: accumulator column of the W3 half
      int got = 0;
      if (lane == 0) got = mbar_wait<true>(&tfull_bar[acc], acc_phase, abort_flag, P.wait_ns) ? 1 : 0;
      got = __shfl_sync(kFull, got, 0);
      if (!got) {
        if (lane == 0) {
          record_error(P.status, kErrTimeout, 203, (int32_t)blockIdx.x, tile);
          s_abort = 1;
        }
        break;
      }
      tc_fence_after();
      const bool valid = r < kTR && ti.mt * kTR + r < ti.m;
      // bf16 outputs of a warp whose 32 rows all belong to the group go out as one
      // TMA block store; a group's ragged last rows are stored row by row.
      const bool use_tma = EPI != kLogits && (!kMx || EPI == kLinear) && F.tma_out && q * 32 + 32 <= kTR &&
                           ti.mt * kTR + q * 32 + 32 <= ti.m;
      const int64_t grow = (int64_t)ti.a_row0 + r;
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      // H tiles (GELU / SwiGLU) are stored as bf16 for the next GEMM; gate-scaled
      // expert outputs (linear epilogue) stay fp32 until the combine's single rounding.
      const int64_t out_off =
          grow * F.ld_out + (int64_t)ti.g * F.out_col_group + (int64_t)ti.nt * kOutCols + col_shift;
      const int32_t ox0 = (int32_t)((int64_t)ti.g * F.out_col_group + (int64_t)ti.nt * kOutCols + col_shift);
      const int32_t oy = ti.a_row0 + q * 32;
      const CUtensorMap* omap = ti.fam == 0 ? &o0 : &o1;
      const int64_t bcol0 = (int64_t)ti.nt * kOutCols + col_shift;
      const __nv_bfloat16* bias = F.bias ? F.bias + (int64_t)ti.g * F.bias_group : nullptr;
      float gate = 1.f;
      if (EPI == kLinear && F.row_gate && valid) gate = F.row_gate[grow];

      // one 32-column chunk: registers v (and u, the W3 half for SwiGLU) -> outputs.
      // bf16 results are packed in place (pk), fp32 results overwrite v.
      auto finish_chunk = [&](uint32_t(&v)[32], uint32_t(&u)[32], int c) {
        if constexpr (kMx && EPI != kLinear) {
          // MXFP8 H: the chunk's 32 columns of the row are one MX block, stored as 32
          // E4M3 codes and their E8M0 scale byte
          float hv[32];
          if (EPI == kSwiglu) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 h = act::silu_mul2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                              make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])));
              hv[2 * i] = h.x;
              hv[2 * i + 1] = h.y;
            }
          } else {
            uint4 braw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                             make_uint4(0, 0, 0, 0)};
            if (bias) {  // routed experts: one bias vector
              const uint4* bp = reinterpret_cast<const uint4*>(bias + bcol0 + c);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) braw[q4] = __ldg(bp + q4);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t bw = (&braw[i >> 2].x)[i & 3];  // bf16x2: low half = column 2i
              const float2 a = __fadd2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                          make_float2(__uint_as_float(bw << 16), __uint_as_float(bw & 0xFFFF0000u)));
              const float2 g = act::gelu2_as7128(a);
              hv[2 * i] = g.x;
              hv[2 * i + 1] = g.y;
            }
          }
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
          const uint32_t sb = mx::scale_byte(amax);
          const float inv = mx::inv_scale(sb);
          uint32_t q8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            q8[i] = mx::e4m3x4(hv[4 * i] * inv, hv[4 * i + 1] * inv, hv[4 * i + 2] * inv, hv[4 * i + 3] * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(F.out) + out_off + c);
            dst[0] = make_uint4(q8[0], q8[1], q8[2], q8[3]);
            dst[1] = make_uint4(q8[4], q8[5], q8[6], q8[7]);
            F.out_scale[grow * F.out_scale_ld + (bcol0 + c) / 32] = (uint8_t)sb;
          }
          return;
        }
        uint32_t pk[16];
        if (EPI == kSwiglu) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // SiLU(a) * u, two columns per packed op
            const float2 h = act::silu_mul2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                            make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])));
            const __nv_bfloat162 hb = __floats2bfloat162_rn(h.x, h.y);
            pk[i] = *reinterpret_cast<const uint32_t*>(&hb);
          }
        } else {
          // bias: one bf16 vector (common case) kept packed, or a sum of several added in place
          uint4 braw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                           make_uint4(0, 0, 0, 0)};
          const bool one_bias = bias && F.bias_nsum == 1;
          if (one_bias) {
            const uint4* bp = reinterpret_cast<const uint4*>(bias + bcol0 + c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) braw[q4] = __ldg(bp + q4);
          } else if (bias) {
            for (int s = 0; s < F.bias_nsum; ++s) {
              const uint4* bp = reinterpret_cast<const uint4*>(bias + s * F.bias_sum_stride + bcol0 + c);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                float bv[8];
                Vec16<__nv_bfloat16>::unpack(__ldg(bp + q4), bv);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[8 * q4 + i] = __float_as_uint(__uint_as_float(v[8 * q4 + i]) + bv[i]);
              }
            }
          }
          if (EPI == kLogits && F.bias_f32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int64_t col = bcol0 + c + i;
              if (col < F.n_valid) v[i] = __float_as_uint(__uint_as_float(v[i]) + __ldg(F.bias_f32 + col));
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0 = __uint_as_float(v[2 * i]), a1 = __uint_as_float(v[2 * i + 1]);
            if (EPI == kGelu) {
              float2 a = make_float2(a0, a1);
              if (one_bias) {
                const uint32_t bw = (&braw[i >> 2].x)[i & 3];  // bf16x2: low half = column 2i
                a = __fadd2_rn(a, make_float2(__uint_as_float(bw << 16), __uint_as_float(bw & 0xFFFF0000u)));
              }
              const float2 g = act::gelu2_as7128(a);
              const __nv_bfloat162 hb = __floats2bfloat162_rn(g.x, g.y);
              pk[i] = *reinterpret_cast<const uint32_t*>(&hb);
              continue;
            }
            float2 a = make_float2(a0, a1);
            if (one_bias) {
              const uint32_t bw = (&braw[i >> 2].x)[i & 3];  // bf16x2: low half = column 2i
              a = __fadd2_rn(a, make_float2(__uint_as_float(bw << 16), __uint_as_float(bw & 0xFFFF0000u)));
            }
            if (EPI == kLinear) a = __fmul2_rn(a, make_float2(gate, gate));
            v[2 * i] = __float_as_uint(a.x);
            v[2 * i + 1] = __float_as_uint(a.y);
          }
        }
        if (use_tma) {
          // 64-byte rows through the staging block: row `lane`, 16-byte chunk j stored at
          // chunk j ^ ((row >> 1) & 3) (64-byte swizzle). bf16: one 32-column block;
          // fp32: two 16-column blocks.
#pragma unroll
          for (int h = 0; h < (EPI == kLinear ? 2 : 1); ++h) {
            if (lane == 0 && store_pending) bulk_wait_read0();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 val = EPI == kLinear
                                    ? make_uint4(v[16 * h + 4 * j], v[16 * h + 4 * j + 1], v[16 * h + 4 * j + 2],
                                                 v[16 * h + 4 * j + 3])
                                    : make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              *reinterpret_cast<uint4*>(staging + lane * 64 + 16 * (j ^ ((lane >> 1) & 3))) = val;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(omap, staging, ox0 + c + 16 * h, oy);
              bulk_commit();
            }
            store_pending = true;
          }
        } else if (valid && EPI == kLogits) {
          float* dst = static_cast<float*>(F.out) + out_off + c;
          const int64_t col0 = bcol0 + c;
          if (col0 + 32 <= F.n_valid && (F.ld_out & 3) == 0) {  // rows 16-byte aligned
#pragma unroll
            for (int i = 0; i < 8; ++i)
              reinterpret_cast<uint4*>(dst)[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < F.n_valid) dst[i] = __uint_as_float(v[i]);
          }
        } else if (valid) {
          if (EPI == kLinear) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(F.out) + out_off + c);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(F.out) + out_off + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      };

      // chunks c = part*32, part*32 + 32*(kEpiWarps/4), ... (none for quadrants past the tile's rows)
      uint32_t va[32], ua[32];
      for (int c = part * 32; q * 32 < kTR && c < out_cols; c += 32 * (kEpiWarps / 4)) {
        tmem_ld32(tbase + (uint32_t)c, va);
        if (EPI == kSwiglu) tmem_ld32(tbase + (uint32_t)(u_cols + c), ua);
        tmem_ld_wait(va);
        if (EPI == kSwiglu) reg_fence(ua);
        finish_chunk(va, ua, c);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (!PAIR || rank == 0)
          mbar_arrive(&tempty_bar[acc]);
        else  // the leader's MMAs wait for both halves of the accumulator to be drained
          mbar_arrive_remote(mapa_shared(smem_u32(&tempty_bar[acc]), 0u));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0 && store_pending) bulk_wait0();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // PAIR: neither CTA leaves while the other may still signal its barriers
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_t<PAIR>(tmem_base, C::kTmemCols);
  }
}

// ---- host side ---------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D matrix [rows, cols] row-major, box = box_cols x box_rows.
bool make_map_ex(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows,
                 CUtensorMapDataType dt, int elem_bytes, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || !ptr || rows < 1 || cols < box_cols) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand tiles: bf16, 64 columns (one 128-byte swizzle atom) x box_rows rows.
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  return make_map_ex(m, ptr, rows, cols, BK, box_rows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output blocks of 32 rows x 64 bytes, 64-byte swizzle (the epilogue staging layout):
// bf16 32 columns, or fp32 16 columns.
bool make_out_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols) {
  return make_map_ex(m, ptr, rows, cols, 32, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B);
}
bool make_out_map_f32(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols) {
  return make_map_ex(m, ptr, rows, cols, 16, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Bound on each pipeline wait of the single-CTA grouped GEMM: 2 s, or the value of
// the environment variable MOE_GEMM_WAIT_LIMIT_NS when it is set (read at every
// launch; lets a test make the waits run out and check that the kernel reports
// MOE_ERR_TIMEOUT and tears down cleanly). The teardown's waits for copies and MMAs
// in flight, and every wait of the CTA-pair form, keep the 2 s bound.
unsigned long long wait_limit_ns() {
  const char* v = std::getenv("MOE_GEMM_WAIT_LIMIT_NS");
  if (!v || !*v) return kTimeoutNs;
  char* end = nullptr;
  const unsigned long long n = std::strtoull(v, &end, 10);
  return (end && *end == 0 && n > 0 && n <= kTimeoutNs) ? n : kTimeoutNs;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// grid_cap > 0: at most this many CTAs (the rest of the SMs stay free for other work).
template <int BN, int EPI, int MXR = 0>
cudaError_t launch_t(const CUtensorMap (&maps)[8], const Params& P, int64_t max_tiles, cudaStream_t st,
                     int64_t grid_cap = 0) {
  using C = Cfg<BN, false, MXR, !(MXR != 0 && EPI != kLinear)>;
  auto kern = grouped_gemm_kernel<BN, EPI, false, MXR>;
  static cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (attr != cudaSuccess) return attr;
  int64_t grid = max_tiles < num_sms() ? max_tiles : num_sms();
  if (grid_cap > 0 && grid > grid_cap) grid = grid_cap;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), C::kSmem, st, maps[0], maps[1], maps[2], maps[3],
                    maps[4], maps[5], maps[6], maps[7], P);
}

// CTA-pair form: clusters of two CTAs, one cluster per pair tile up to the number of
// clusters the GPU holds at once (persistent), launched with the same dependent-launch
// attribute as the single-CTA form.
template <int BN, int EPI>
cudaError_t launch_pair_t(const CUtensorMap (&maps)[8], const Params& P, int64_t max_pair_tiles, cudaStream_t st,
                          int64_t grid_cap = 0) {
  using C = Cfg<BN, true>;
  auto kern = grouped_gemm_kernel<BN, EPI, true>;
  static cudaError_t attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (attr != cudaSuccess) return attr;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  static int resident = [&]() {
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3((unsigned)num_sms());
    q.numAttrs = 1;  // cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = num_sms() / 2;
    }
    return n;
  }();
  int64_t clusters = max_pair_tiles < resident ? max_pair_tiles : resident;
  if (grid_cap > 0 && 2 * clusters > grid_cap) clusters = grid_cap / 2 > 0 ? grid_cap / 2 : 1;
  if (clusters <= 0) return cudaSuccess;
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], P);
}

template <int EPI>
cudaError_t launch_bn(int bn, const CUtensorMap (&maps)[8], const Params& P, int64_t max_tiles, cudaStream_t st,
                      int64_t grid_cap = 0) {
  switch (bn) {
    case 256: return launch_t<256, EPI>(maps, P, max_tiles, st, grid_cap);
    case 128: return launch_t<128, EPI>(maps, P, max_tiles, st, grid_cap);
    default: return launch_t<64, EPI>(maps, P, max_tiles, st, grid_cap);
  }
}

// MXFP8 form: 128-column tiles of 32 A rows when the experts average at most 32 rows
// (decode batches: the weight stream is the work, A is a 4 KB box), else 128.
template <int EPI>
cudaError_t launch_mx(int rows, const CUtensorMap (&maps)[8], const Params& P, int64_t max_tiles, cudaStream_t st,
                      int64_t grid_cap) {
  return rows == 32 ? launch_t<128, EPI, 32>(maps, P, max_tiles, st, grid_cap)
                    : launch_t<128, EPI, 128>(maps, P, max_tiles, st, grid_cap);
}

// E4M3 codes of a matrix [rows, K] (bytes): 128-byte rows (128 codes, one stage) x
// box_rows, 128-byte swizzle (the MMA's operand layout, as for 64 bf16).
bool make_code_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  return make_map_ex(m, ptr, rows, cols, 128, box_rows, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// Largest tile width BN in {256, 128, 64} whose output width (BN, or BN/2 for
// SwiGLU) divides every listed column count.
int pick_bn(bool swiglu, int64_t c0, int64_t c1) {
  for (int bn : {256, 128, 64}) {
    const int oc = swiglu ? bn / 2 : bn;
    if (c0 % oc == 0 && (c1 <= 0 || c1 % oc == 0)) return bn;
  }
  return 0;
}

}  // namespace tc

bool tc_gemm_available() { return tc::encode_fn() != nullptr; }

// Router logits on the tensor cores: N token rows against the E router rows
// (zero-filled past E by the tensor map), fp32 out. splits = 1: logits + bias into
// `out` [N, E]. splits > 1: the K range is cut into `splits` groups of equal
// length, group g writing its partial sums (no bias) to slab g of `out`
// ([splits][N][E]); the routing kernel adds the slabs in order and the bias.
cudaError_t launch_router_logits_tc(const Plan& p, const void* x, const void* w_router, const float* logit_bias,
                                    float* out, int splits, int32_t* status, cudaStream_t st) {
  using namespace tc;
  const int bn = p.E <= 64 ? 64 : (p.E <= 128 ? 128 : 256);
  const int64_t kb = p.d / BK;
  if (splits < 1 || kb % splits) return cudaErrorInvalidValue;
  // 256-wide tiles run on CTA pairs (each CTA stages half of W_r's tile: shallower
  // stages, so a deeper ring of x in flight) once the batch has two 128-row tiles
  const bool pair = bn == 256 && p.N > BM;
  CUtensorMap maps[8];
  if (!make_map(&maps[0], x, p.N, p.d, BM)) return cudaErrorInvalidValue;
  if (!make_map(&maps[1], w_router, p.E, p.d, pair ? bn / 2 : bn)) return cudaErrorInvalidValue;
  for (int i = 2; i < 8; ++i) maps[i] = maps[0];
  Params P{};
  Family& f0 = P.fam[0];
  f0.groups = splits;
  f0.m_fixed = (int32_t)p.N;
  f0.n_tiles = (int32_t)ceil_div(p.E, bn);
  f0.k_blocks = f0.kseg_blocks = (int32_t)(kb / splits);
  f0.k_group = (int32_t)(kb / splits);
  f0.a_map = 0;
  f0.b_map = 1;
  f0.b3_map = 1;
  f0.out = out;
  f0.ld_out = p.E;
  f0.out_col_group = p.N * p.E;  // slab g
  f0.bias_f32 = splits == 1 ? logit_bias : nullptr;
  f0.n_valid = p.E;
  P.expert_off = nullptr;
  P.status = status;
  P.wait_ns = pair ? kTimeoutNs : wait_limit_ns();  // the pair form keeps the full bound
  if (pair) return launch_pair_t<256, kLogits>(maps, P, ceil_div(p.N, 2 * BM) * f0.n_tiles * splits, st);
  return launch_bn<kLogits>(bn, maps, P, ceil_div(p.N, BM) * f0.n_tiles * splits, st);
}

// The down-projection runs on CTA pairs (256-row tiles, half of B per CTA) with
// 256-wide tiles once the routed experts average at least eight 128-row tiles each;
// smaller batches keep 128-row tiles, whose ragged last tile wastes half as much: an
// expert's odd last 128-row tile costs a whole pair tile, which at four tiles per expert
// (the 16384-token, 256-expert layer) is ~22 % of the tiles against ~11 % (measured
// there: 4.08-4.12 ms on pairs, 3.99 ms on single CTAs). The up-projection stays on
// single CTAs: its epilogue, which pairs do not shorten, bounds it at short K.
bool use_pair_tiles(const Plan& p, int bn) {
  const int64_t R = p.max_rows > 0 ? p.max_rows : 1;
  return bn == 256 && R >= (int64_t)8 * tc::BM * p.E;
}
// The up-projection runs on CTA pairs with 256-wide tiles when the experts' rows fill
// 256-row pair tiles: each CTA stages half of B (32 KB stages instead of 48 KB, six in
// flight instead of four) and the pair shares one copy of each B tile. Measured on B300:
// the 4096-token, 8-expert layer (8 row tiles per expert) 1530 -> 1414 us; expert choice
// with C = 512 (no ragged tile) 7874 -> 7561 us; the 16384-token, 256-expert token-choice
// layer (4-5 ragged tiles per expert, where an odd last 128-row tile costs a pair tile)
// 9043 -> 9108 us, so token choice takes pairs only from 8 tiles per expert.
bool use_pair_up(const Plan& p, int bn) {
  if (bn != 256) return false;
  if (p.ec) return p.cap >= 8 * tc::BM || (p.cap >= 4 * tc::BM && p.cap % (2 * tc::BM) == 0);
  const int64_t R = p.max_rows > 0 ? p.max_rows : 1;
  return R >= (int64_t)8 * tc::BM * p.E;
}

namespace {

// The routed experts of an MXFP8 layer (kind::mxf8f6f4): xp holds the permuted rows'
// E4M3 codes [R, d] and their E8M0 scales [R, d / 32] (mx::scale_offset), H is written
// and read back the same way ([R, F] codes, [R, F / 32] scales), the weights are codes
// and scales. The up-projection quantises H in its epilogue; the down-projection writes
// gate-scaled fp32 rows like the bf16 form.
cudaError_t launch_ffn_mx(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                          const moe_weights* w, void* h, void* yp, int32_t* status, cudaStream_t st, int part,
                          int64_t grid_cap) {
  using namespace tc;
  const int64_t R = p.max_rows > 0 ? p.max_rows : 1;
  const int rows = R <= 32 * p.E ? 32 : 128;  // A rows per tile
  const uint8_t* xq = static_cast<const uint8_t*>(xp);
  uint8_t* h8 = static_cast<uint8_t*>(h);
  if (part & 1) {
    const int brows = p.swiglu ? 64 : 128;  // B rows per map copy (W1 and W3 halves for SwiGLU)
    CUtensorMap maps[8];
    bool ok = make_code_map(&maps[0], xq, R, p.d, rows) && make_code_map(&maps[2], w->w1, p.E * p.F, p.d, brows);
    if (p.swiglu) ok = ok && make_code_map(&maps[3], w->w3, p.E * p.F, p.d, brows);
    if (!ok) return cudaErrorInvalidValue;
    for (int i : {1, 4, 5, 6, 7}) maps[i] = maps[0];
    if (!p.swiglu) maps[3] = maps[0];
    Params P{};
    Family& f = P.fam[0];
    f.groups = (int32_t)p.E;
    f.m_from_off = 1;
    f.n_tiles = (int32_t)(p.F / brows);
    f.k_blocks = f.kseg_blocks = (int32_t)(p.d / (128 * mx_atoms(rows)));
    f.b_rows_group = (int32_t)p.F;
    f.a_map = 0;
    f.b_map = 2;
    f.b3_map = 3;
    f.out = h8;
    f.ld_out = p.F;
    f.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->b1 : nullptr);
    f.bias_group = p.F;
    f.bias_nsum = p.bias ? 1 : 0;
    f.a_rows = (int32_t)R;
    f.a_scale = xq + mx::scale_offset(R, p.d);
    f.a_scale_ld = p.d / 32;
    f.b_scale = w->w1_scale;
    f.b3_scale = w->w3_scale;
    f.scale_ld = p.d / 32;
    f.out_scale = h8 + mx::scale_offset(R, p.F);
    f.out_scale_ld = p.F / 32;
    P.expert_off = expert_off;
    P.status = status;
    P.wait_ns = wait_limit_ns();
    const int64_t max_tiles = (R / rows + p.E) * f.n_tiles;
    const cudaError_t err = p.swiglu ? launch_mx<kSwiglu>(rows, maps, P, max_tiles, st, grid_cap)
                                     : launch_mx<kGelu>(rows, maps, P, max_tiles, st, grid_cap);
    if (err != cudaSuccess) return err;
  }
  if (part & 2) {
    CUtensorMap maps[8];
    if (!make_code_map(&maps[0], h8, R, p.F, rows) || !make_code_map(&maps[2], w->w2, p.E * p.d, p.F, 128) ||
        !make_out_map_f32(&maps[6], yp, R, p.d))
      return cudaErrorInvalidValue;
    for (int i : {1, 3, 4, 5, 7}) maps[i] = maps[0];
    Params P{};
    Family& f = P.fam[0];
    f.tma_out = 1;
    f.groups = (int32_t)p.E;
    f.m_from_off = 1;
    f.n_tiles = (int32_t)(p.d / 128);
    f.k_blocks = f.kseg_blocks = (int32_t)(p.F / (128 * mx_atoms(rows)));
    f.b_rows_group = (int32_t)p.d;
    f.a_map = 0;
    f.b_map = 2;
    f.b3_map = 2;
    f.out = yp;
    f.ld_out = p.d;
    f.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->b2 : nullptr);
    f.bias_group = p.d;
    f.bias_nsum = p.bias ? 1 : 0;
    f.row_gate = row_gate;
    f.a_rows = (int32_t)R;
    f.a_scale = h8 + mx::scale_offset(R, p.F);
    f.a_scale_ld = p.F / 32;
    f.b_scale = w->w2_scale;
    f.scale_ld = p.F / 32;
    P.expert_off = expert_off;
    P.status = status;
    P.wait_ns = wait_limit_ns();
    const cudaError_t err = launch_mx<kLinear>(rows, maps, P, (R / rows + p.E) * f.n_tiles, st, grid_cap);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace

// part: bit 0 = up-projections (routed + shared), bit 1 = down-projections.
// gather_rows non-null: the routed up-projection reads its A rows straight from x
// (row r of the expert-contiguous order is x[gather_rows[r]]) with tile::gather4, and
// xp is not used. MXFP8 layers: the routed experts run in the MXFP8 form, the shared
// experts (bf16 weights) in launches of their own.
cudaError_t launch_ffn_bf16(const Plan& p, const void* xp, const int32_t* expert_off, const float* row_gate,
                            const void* x, const moe_weights* w, void* h, void* hs, void* yp, void* ys,
                            int32_t* status, cudaStream_t st, int part, const int32_t* gather_rows, int families,
                            int64_t grid_cap) {
  using namespace tc;
  if (p.fp8w) {
    if (families & kRoutedFamily) {
      const cudaError_t err = launch_ffn_mx(p, xp, expert_off, row_gate, w, h, yp, status, st, part, grid_cap);
      if (err != cudaSuccess) return err;
    }
    if (!(families & kSharedFamily) || p.S == 0) return cudaSuccess;
    Plan q = p;
    q.fp8w = false;
    return launch_ffn_bf16(q, xp, expert_off, row_gate, x, w, h, hs, yp, ys, status, st, part, nullptr,
                           kSharedFamily, grid_cap);
  }
  const int64_t R = p.max_rows > 0 ? p.max_rows : 1;
  if (part & 1) {
    const int bn = pick_bn(p.swiglu, p.F, p.S > 0 ? p.Fs : 0);
    if (!bn) return cudaErrorInvalidValue;
    const bool pair = !gather_rows && use_pair_up(p, bn);
    const int oc = p.swiglu ? bn / 2 : bn;
    const int brows = p.swiglu || pair ? bn / 2 : bn;
    CUtensorMap maps[8];
    // (a launch of the shared experts alone never reads the routed A map: any valid map)
    const bool ok_a = !(families & kRoutedFamily) ? make_map(&maps[0], x, p.N, p.d, BM)
                      : gather_rows ? make_map_ex(&maps[0], x, p.N, p.d, BK, 1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                                  CU_TENSOR_MAP_SWIZZLE_128B)
                                    : make_map(&maps[0], xp, R, p.d, BM);
    if (!ok_a) return cudaErrorInvalidValue;
    for (int i = 1; i < 8; ++i) maps[i] = maps[0];  // unused slots hold a valid map
    bool ok = (families & kRoutedFamily) ? make_map(&maps[2], w->w1, p.E * p.F, p.d, brows) : true;
    if (p.swiglu && (families & kRoutedFamily)) ok = ok && make_map(&maps[3], w->w3, p.E * p.F, p.d, brows);
    if (p.S > 0) {
      ok = ok && make_map(&maps[1], x, p.N, p.d, BM) && make_map(&maps[4], w->ws1, p.S * p.Fs, p.d, brows);
      if (p.swiglu) ok = ok && make_map(&maps[5], w->ws3, p.S * p.Fs, p.d, brows);
    }
    if (families & kRoutedFamily) ok = ok && make_out_map(&maps[6], h, R, p.F);
    if (p.S > 0) ok = ok && make_out_map(&maps[7], hs, p.N, p.S * p.Fs);
    if (!ok) return cudaErrorInvalidValue;
    Params P{};
    Family& f0 = P.fam[0];
    f0.tma_out = 1;
    P.fam[1].tma_out = p.S > 0 ? 1 : 0;
    f0.groups = (int32_t)p.E;
    f0.m_from_off = 1;
    f0.n_tiles = (int32_t)(p.F / oc);
    f0.k_blocks = f0.kseg_blocks = (int32_t)(p.d / BK);
    f0.b_rows_group = (int32_t)p.F;
    f0.a_map = 0;
    f0.b_map = 2;
    f0.b3_map = 3;
    f0.out = h;
    f0.ld_out = p.F;
    f0.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->b1 : nullptr);
    f0.bias_group = p.F;
    f0.bias_nsum = p.bias ? 1 : 0;
    f0.gather_rows = gather_rows;
    f0.gather_n = (int32_t)p.N;
    if (p.S > 0) {
      Family& f1 = P.fam[1];
      f1.groups = (int32_t)p.S;
      f1.m_fixed = (int32_t)p.N;
      f1.n_tiles = (int32_t)(p.Fs / oc);
      f1.k_blocks = f1.kseg_blocks = (int32_t)(p.d / BK);
      f1.b_rows_group = (int32_t)p.Fs;
      f1.a_map = 1;
      f1.b_map = 4;
      f1.b3_map = 5;
      f1.out = hs;
      f1.ld_out = p.S * p.Fs;
      f1.out_col_group = p.Fs;
      f1.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->bs1 : nullptr);
      f1.bias_group = p.Fs;
      f1.bias_nsum = p.bias ? 1 : 0;
    }
    P.expert_off = expert_off;
    P.status = status;
    P.wait_ns = pair ? kTimeoutNs : wait_limit_ns();  // the pair form keeps the full bound
    if (!(families & kRoutedFamily)) f0.groups = 0;
    if (!(families & kSharedFamily)) P.fam[1].groups = 0;
    if (pair) {
      const int64_t max_pairs = (f0.groups ? (R / (2 * BM) + p.E) * f0.n_tiles : 0) +
                                (P.fam[1].groups ? p.S * ceil_div(p.N, 2 * BM) * P.fam[1].n_tiles : 0);
      if (max_pairs > 0) {
        const cudaError_t err = p.swiglu ? launch_pair_t<256, kSwiglu>(maps, P, max_pairs, st, grid_cap)
                                         : launch_pair_t<256, kGelu>(maps, P, max_pairs, st, grid_cap);
        if (err != cudaSuccess) return err;
      }
    } else {
      const int64_t max_tiles = (f0.groups ? (R / BM + p.E) * f0.n_tiles : 0) +
                                (P.fam[1].groups ? p.S * ceil_div(p.N, BM) * P.fam[1].n_tiles : 0);
      if (max_tiles > 0) {
        const cudaError_t err = p.swiglu ? launch_bn<kSwiglu>(bn, maps, P, max_tiles, st, grid_cap)
                                         : launch_bn<kGelu>(bn, maps, P, max_tiles, st, grid_cap);
        if (err != cudaSuccess) return err;
      }
    }
  }
  if (part & 2) {
    const int bn = pick_bn(false, p.d, 0);
    if (!bn) return cudaErrorInvalidValue;
    const bool pair = use_pair_tiles(p, bn);
    const int brows = pair ? bn / 2 : bn;
    CUtensorMap maps[8];
    // (a launch of the shared experts alone never reads the routed maps: any valid map)
    const bool routed = (families & kRoutedFamily) != 0;
    if (!(routed ? make_map(&maps[0], h, R, p.F, BM) : make_map(&maps[0], hs, p.N, p.S * p.Fs, BM)))
      return cudaErrorInvalidValue;
    for (int i = 1; i < 8; ++i) maps[i] = maps[0];
    bool ok = routed ? make_map(&maps[2], w->w2, p.E * p.d, p.F, brows) : true;
    if (p.S > 0)
      ok = ok && make_map(&maps[1], hs, p.N, p.S * p.Fs, BM) && make_map(&maps[3], w->ws2, p.S * p.d, p.Fs, brows);
    if (routed) ok = ok && make_out_map_f32(&maps[6], yp, R, p.d);
    if (p.S > 0) ok = ok && make_out_map_f32(&maps[7], ys, p.N, p.d);
    if (!ok) return cudaErrorInvalidValue;
    Params P{};
    Family& f0 = P.fam[0];
    f0.tma_out = 1;
    P.fam[1].tma_out = p.S > 0 ? 1 : 0;
    f0.groups = (int32_t)p.E;
    f0.m_from_off = 1;
    f0.n_tiles = (int32_t)(p.d / bn);
    f0.k_blocks = f0.kseg_blocks = (int32_t)(p.F / BK);
    f0.b_rows_group = (int32_t)p.d;
    f0.a_map = 0;
    f0.b_map = 2;
    f0.b3_map = 2;
    f0.out = yp;
    f0.ld_out = p.d;
    f0.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->b2 : nullptr);
    f0.bias_group = p.d;
    f0.bias_nsum = p.bias ? 1 : 0;
    f0.row_gate = row_gate;
    if (p.S > 0) {
      Family& f1 = P.fam[1];
      f1.groups = 1;
      f1.m_fixed = (int32_t)p.N;
      f1.n_tiles = (int32_t)(p.d / bn);
      f1.k_blocks = (int32_t)(p.S * p.Fs / BK);
      f1.kseg_blocks = (int32_t)(p.Fs / BK);
      f1.b_rows_kseg = (int32_t)p.d;
      f1.a_map = 1;
      f1.b_map = 3;
      f1.b3_map = 3;
      f1.out = ys;
      f1.ld_out = p.d;
      f1.bias = static_cast<const __nv_bfloat16*>(p.bias ? w->bs2 : nullptr);
      f1.bias_sum_stride = p.d;
      f1.bias_nsum = p.bias ? (int32_t)p.S : 0;
    }
    P.expert_off = expert_off;
    P.status = status;
    P.wait_ns = pair ? kTimeoutNs : wait_limit_ns();  // the pair form keeps the full bound
    if (!routed) f0.groups = 0;
    if (!(families & kSharedFamily)) P.fam[1].groups = 0;
    cudaError_t err = cudaSuccess;
    if (pair) {
      const int64_t max_pairs = (f0.groups ? (R / (2 * BM) + p.E) * f0.n_tiles : 0) +
                                (P.fam[1].groups ? ceil_div(p.N, 2 * BM) * P.fam[1].n_tiles : 0);
      if (max_pairs > 0) err = launch_pair_t<256, kLinear>(maps, P, max_pairs, st, grid_cap);
    } else {
      const int64_t tiles = (f0.groups ? (R / BM + p.E) * f0.n_tiles : 0) +
                            (P.fam[1].groups ? ceil_div(p.N, BM) * P.fam[1].n_tiles : 0);
      if (tiles > 0) err = launch_bn<kLinear>(bn, maps, P, tiles, st, grid_cap);
    }
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace moe
