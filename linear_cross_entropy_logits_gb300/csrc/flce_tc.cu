// Tensor-core GEMMs of the fused linear cross entropy for sm_103a: tcgen05.mma with
// fp32 accumulators in tensor memory (TMEM), operands staged in shared memory by TMA
// (cp.async.bulk.tensor, 128-byte swizzle), warp-specialised and persistent.
//
// One kernel template serves the three products of the method:
//   FWD: S = Xc W^T (K = H). The epilogue never writes S: per row and per 256-column
//        vocabulary tile it keeps the max, the sum of the exponentials, the lowest-index
//        argmax and the target logit, and writes exp(s) (row-reference form) or
//        exp(s - tile max) (per-tile form), in the input dtype, from registers into the
//        chunk slab, from which the gradient is formed once the row's lse is known.
//   DX:  dX[idx] = cbar * G W (K = V): tiles, optionally split in up to four K ranges,
//        added by TMA reduce-add into two zeroed fp32 chunk buffers (at most two adds per
//        element, onto zero), then summed and scattered to the dX rows through the
//        compaction index by k_dx_store.
//   DW:  dW += cbar * G^T Xc (K = chunk rows), added into the destination by TMA
//        reduce-add from the single CTA pair that owns each tile (one add per element per
//        launch: deterministic).
//   BWD: the DX and DW work of a chunk in one persistent launch (k_gemm_bwd): the pairs
//        draw work items (dX items first, then dW tiles) from a device-wide queue, so that
//        dW fills dX's last wave; results bit-identical to two launches.
// The three products are the logits, grad_input and grad_weight GEMMs that the pages'
// op runs in its forward ("Liger-Kernel PR #1554: skip ignore_index rows", Summary); dW is
// accumulated straight into the caller's buffer with no [V,H] temporary ("Reduce FLCE
// weight-gradient allocation overhead across FP16, BF16, and FP32", Proposed direction).
//
// Launch shape: clusters of 2 CTAs (one CTA pair = two SMs of a TPC), one CTA per SM,
// persistent over pair tiles of 256 (M) x 256 or 256 x 512 (N). The pair runs
// tcgen05.mma.cta_group::2 with M = 256 and N = 256: each CTA stages its own 128 rows of A
// and one half (128 rows) of each B sub-tile, and holds its 128-row fp32 accumulator in its
// own TMEM. 256 x 256 tiles (6 stages of 32 KB) keep two accumulators, so a tile's
// epilogue overlaps the next tile's mainloop; 256 x 512 tiles (4 stages of 48 KB) issue two
// MMAs per staged A block, a quarter less operand traffic per FLOP, with one 512-column
// accumulator whose epilogue is exposed.
//
// Warp roles (320 threads per CTA):
//   warp 0        TMA producer (one thread) in both CTAs; the peer's copies complete on
//                 the leader's "full" barrier, which the leader arms for both halves
//   warp 1        TMEM allocator (both CTAs) and, in the leader CTA, the MMA issuer (one
//                 thread); its commits arrive on both CTAs' "empty" / "tmem full" barriers
//   warps 2..9    epilogue in both CTAs (2..5 only on 256 x 256 tiles); warp w reads TMEM
//                 lanes 32*(w%4) .. +31 of sub-tile (w-2)/4, and both CTAs' epilogues
//                 arrive on the leader's "tmem empty" barrier
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// FLCE_ERR_TIMEOUT, tells its peer, and both leave their loops; before TMEM is freed the
// pair reconciles the copies each CTA issued against the leader's barriers and waits
// (bounded) for them and for the MMAs in flight.
#include <cuda.h>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "flce_internal.cuh"

namespace flce {
namespace tc {

constexpr int BM = 128;                            // rows of A per CTA (pair tile M = 256)
constexpr int BN = 256;                            // N of one MMA (each CTA holds BN/2 of B)
constexpr int BK = 64;

enum Mode { FWD = 0, DX = 1, DW = 2 };

// Pair tile width in 256-column sub-tiles. NB = 2: a 256 x 512 pair tile whose two MMAs
// per K step share the A stage (37% more FLOPs per operand byte than 256 x 256; the GEMMs
// are bound by the operand feed), with one 512-column TMEM accumulator and eight epilogue
// warps (one per TMEM lane quadrant and sub-tile). NB = 1: 256 x 256 tiles with two
// 256-column accumulators, so that a tile's epilogue overlaps the next tile's mainloop.
// The forward takes NB = 2 when H >= FWD_WIDE_MIN_H and NB = 1 below (a short K cannot
// hide the exposed epilogue of the single accumulator); dX takes NB = 2 (K = V, the
// epilogue is negligible); dW takes NB = 2 when a chunk holds at least DW_WIDE_MIN_ROWS
// rows and NB = 1 below that. At 2048 to 4096 rows the two dW shapes run at the same rate
// (the wide tile's exposed reduce-add epilogue against the narrow one's operand feed), and
// the wide one lets dW share the merged dX + dW launch (2.5% faster on the large-vocab
// head at 2688-row chunks; outputs bit-identical).
// DW_WIDE_MIN_ROWS, FWD_WIDE_MIN_H (flce_internal.cuh): the forward takes the wide tile
// from H = 4096 on, where its K loop is long enough that the wide tile's smaller operand
// traffic per FLOP outweighs its exposed epilogue (measured 1% faster at H = 4096, in short
// and in power-capped runs; 10% slower at H = 2048).
constexpr int A_BYTES = BM * BK * 2;               // 16 KB
constexpr int B_BYTES = (BN / 2) * BK * 2;         // 16 KB per 256-column sub-tile
template <int NB>
__host__ __device__ constexpr int stage_bytes() {
  return A_BYTES + NB * B_BYTES;                   // 32 or 48 KB per CTA
}
// Pipeline depth: 192 KB of stages (6 x 32 KB or 4 x 48 KB), next to the dX / dW epilogue
// staging (the forward stages nothing).
#ifndef FLCE_WIDE_STAGES
#define FLCE_WIDE_STAGES 4
#endif
template <int NB>
__host__ __device__ constexpr int stages_of() {
  return NB == 1 ? 6 : FLCE_WIDE_STAGES;
}
template <int NB>
__host__ __device__ constexpr int nacc_of() {      // TMEM accumulators (512 columns in all)
  return NB == 1 ? 2 : 1;
}
template <int NB>
__host__ __device__ constexpr int epi_warps_of() {
  return 4 * NB;
}
constexpr int MAX_STAGES = 6;
constexpr int BOX_BYTES = 64 * 64 * 2;             // one 64x64 MN-major TMA box (8 KB)
constexpr int NUM_THREADS = 320;                   // producer, MMA, 8 epilogue warps
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_BARS = 2 * MAX_STAGES + 5;       // full, empty, tfull[2], tempty[2], drain
// Epilogue staging of DX / DW: 32 KB, split over the active epilogue warps: 32-row x
// 128-byte buffers (two per warp with four warps, one with eight) that feed TMA
// reduce-adds (the L2 performs dst += tile; no register read-modify-write). The forward
// writes its exp slab straight from registers and stages nothing.
constexpr int EPI_BUF_BYTES = 32 * 128;
constexpr int EPI_BYTES_MIN = 8 * EPI_BUF_BYTES;   // 32 KB
// Epilogue staging of a tile shape: 32 KB, or for the wide tile whatever the stages leave
// (in 2 KB buffers per warp, a multiple of 16 KB).
template <int NB>
__host__ __device__ constexpr int epi_bytes_of() {
  return NB == 1 ? EPI_BYTES_MIN
                 : ((232448 - 1536 - stages_of<NB>() * stage_bytes<NB>()) / 16384) * 16384;
}
template <int NB>
__host__ __device__ constexpr int epi_warp_bytes_of() {  // staging per epilogue warp
  return epi_bytes_of<NB>() / (4 * NB);
}
template <int NB>
__host__ __device__ constexpr int half_bufs_of() {  // 2 KB staging buffers per epilogue warp
  return epi_warp_bytes_of<NB>() / 2048;
}
template <int NB>
__host__ __device__ constexpr int epi_nbuf_of() {
  return 8 / epi_warps_of<NB>();
}
// Staging bytes a launch reserves: none for the forward.
template <int MODE, int NB>
__host__ __device__ constexpr int epi_bytes_m() {
  return MODE == FWD ? 0 : epi_bytes_of<NB>();
}
template <int MODE, int NB>
constexpr int smem_bytes() {
  return stages_of<NB>() * stage_bytes<NB>() + epi_bytes_m<MODE, NB>() + 1024 + 512;
}
static_assert(smem_bytes<DX, 1>() <= 232448 && smem_bytes<DX, 2>() <= 232448, "shared memory per CTA");
static_assert(half_bufs_of<1>() >= 2 && half_bufs_of<2>() >= 2, "epilogue staging buffers");

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
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
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// As mbar_try, but the thread may sleep up to `hint_ns` waiting for the phase (it resumes
// as soon as the phase completes), so waiting warps take no issue slots from the warps
// that feed the tensor cores.
__device__ __forceinline__ bool mbar_try_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Where a CTA gives up: its own abort flag, the peer's (cluster address), the status word.
struct Abort {
  volatile int* flag;
  uint32_t peer_flag;
  int* status;
  uint64_t timeout_ns;
};

// Bounded wait for the phase of `bar` with parity `parity`. Gives up (returning false)
// when this CTA has been told to abort (if honor_abort) or after timeout_ns, in which case
// it raises both CTAs' abort flags and the device status bit.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Abort& ab, bool honor_abort) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (;;) {
    if (mbar_try_sleep(bar, parity, 50000u)) return true;
    if (honor_abort && *ab.flag) return false;
    if (gtimer() - t0 > ab.timeout_ns) {
      *ab.flag = 1;
      st_cluster_u32(ab.peer_flag, 1u);
      atomicOr(ab.status, ST_TIMEOUT);
      return false;
    }
  }
}

// TMA tile load into this CTA's shared memory; completion is counted on `bar`, which may
// be in either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"((uint64_t)map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// dst[box at (x, y)] += smem tile, performed by the TMA unit / L2 (fp32 add).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          (uint64_t)map),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
// Box at (x, y) of the map's tensor = smem tile (clipped at the tensor's extent).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   (uint64_t)map),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N bulk groups of this thread still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), sm100 version bit.
//   K-major operand:  rows of 128 B (64 elements along K), 8-row atoms of 1024 B;
//                     SBO = 1024 (next 8 rows), LBO unused; K steps of 16 = +32 B.
//   MN-major operand: 64 MN-elements per 128-B row, one row per K index, 8-row atoms of
//                     1024 B; SBO = 1024 (next 8 K indices), LBO = 8192 (next 64-wide
//                     MN block = next 64x64 TMA box); K steps of 16 = +2048 B.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulate, A/B format, majors,
// N >> 3 at bit 17, M >> 4 at bit 24 (M = 256: the pair's two 128-row halves).
template <int MODE, typename T>
__device__ __forceinline__ constexpr uint32_t make_idesc() {
  constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  constexpr uint32_t a_mn = MODE == DW ? 1u : 0u;
  constexpr uint32_t b_mn = MODE == FWD ? 0u : 1u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` (same offset) in both CTAs of the pair once all MMAs issued so far are
// complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// Arrive on this CTA's `bar` once all MMAs issued so far are complete.
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; waits for completion so the
// registers are valid on return.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 64 consecutive fp32 columns (two 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
      "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]),
        "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]),
        "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]),
        "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]),
        "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}

// N consecutive fp32 columns (N = 32 or 64), waited for.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 64) tmem_ld64(taddr, r);
  else tmem_ld32(taddr, r);
}

// Columns per TMEM load in the forward epilogue (32 or 64): the block over which a thread
// keeps its row's logits in registers, takes a maximum and may search the argmax.
#ifndef FLCE_FWD_COLS
#define FLCE_FWD_COLS 64
#endif
constexpr int FC = FLCE_FWD_COLS;
static_assert(FC == 32 || FC == 64, "forward epilogue block");

// 2^x by the hardware approximation (ex2.approx.ftz: relative error about 2^-22, results
// below 2^-126 flushed to zero), far finer than the 2^-9 rounding of the 16-bit slab the
// values are stored in; the accurate library exp2f made the epilogue arithmetic-bound.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float x, float y);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *(uint32_t*)&h;
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float x, float y) {
  __half2 h = __floats2half2_rn(x, y);
  return *(uint32_t*)&h;
}

// ------------------------------------------------------------------ tile space
// Pair tiles: m indexes 256-row blocks of the output, n blocks of NB 256-column sub-tiles
// (sub-tile index n * NB + j). nsub = the output's 256-column sub-tiles.
struct TileSpace {
  int mt, nt, nkb, nsub;
};
template <int MODE, int NB>
__device__ __forceinline__ TileSpace tile_space(const CallArgs& a, int rows) {
  TileSpace t;
  if (MODE == FWD) {
    t.mt = cdiv(rows, 2 * BM);
    t.nsub = (int)a.nvt;
    t.nkb = cdiv((int)a.H, BK);
  } else if (MODE == DX) {
    t.mt = cdiv(rows, 2 * BM);
    t.nsub = cdiv((int)a.H, BN);
    t.nkb = cdiv((int)a.V, BK);
  } else {
    t.mt = cdiv((int)a.V, 2 * BM);
    t.nsub = cdiv((int)a.H, BN);
    t.nkb = cdiv(rows, BK);
  }
  t.nt = cdiv(t.nsub, NB);
  return t;
}
// FWD walks m fastest (the pairs in flight share W tiles); DX and DW walk n fastest (the
// pairs in flight share the slab rows / columns).
#ifndef FLCE_FWD_MGROUP
#define FLCE_FWD_MGROUP 16
#endif
// The forward walks its row tiles in groups of FWD_MGROUP (4096 rows): within a group m
// fastest, then n; so the gathered rows a wave needs (a group's Xc, 33 MB) stay in L2
// while W streams, at the price of reading W once per group.
constexpr int FWD_MGROUP = FLCE_FWD_MGROUP;
template <int MODE>
__device__ __forceinline__ void tile_coords(const TileSpace& ts, int tile, int& m, int& n) {
  if (MODE == FWD) {
    if (FWD_MGROUP > 0 && ts.mt > FWD_MGROUP) {
      const int per_group = FWD_MGROUP * ts.nt;
      const int g = tile / per_group, t = tile - g * per_group;
      const int gm = min(FWD_MGROUP, ts.mt - g * FWD_MGROUP);  // rows tiles in this group
      m = g * FWD_MGROUP + t % gm;
      n = t / gm;
    } else {
      m = tile % ts.mt;
      n = tile / ts.mt;
    }
  } else {
    n = tile % ts.nt;
    m = tile / ts.nt;
  }
}

// Work items of one pair: (pair tile, k-block range, split), taken round-robin over the
// pairs so that the pairs in flight walk the same k-blocks in step and share operand tiles
// in L2. FWD and DW take whole tiles. DX (few, long tiles: K = V) may split each tile's K
// range in S <= 4 parts (items ordered split-major) when that fills the last wave better.
// Split s adds its partial sum into fp32 buffer s / 2, zeroed beforehand, so each buffer
// element receives at most two adds onto zero: the result does not depend on their order.
constexpr int DX_MAX_SPLITS = 4;
__device__ __forceinline__ int dx_splits(int ntiles, int npairs, int nkb) {
  // wave efficiency e(S) = ntiles*S / (waves(S)*P); take the smallest S within 2% of the
  // best (fewer splits add fewer partial sums)
  int best = 1;
  float eb = 0.0f;
  float e[DX_MAX_SPLITS + 1];
  for (int S = 1; S <= DX_MAX_SPLITS && S <= nkb; ++S) {
    const int items = ntiles * S, waves = (items + npairs - 1) / npairs;
    e[S] = (float)items / (float)(waves * npairs);
    if (e[S] > eb) eb = e[S];
  }
  for (int S = 1; S <= DX_MAX_SPLITS && S <= nkb; ++S)
    if (e[S] >= 0.98f * eb) {
      best = S;
      break;
    }
  return best;
}
template <int MODE>
struct Items {
  int i, nitems, npairs, ntiles, nkb, S;
  __device__ __forceinline__ Items(int pair, int npairs_, int ntiles_, int nkb_)
      : i(pair), npairs(npairs_), ntiles(ntiles_), nkb(nkb_) {
    S = MODE == DX ? dx_splits(ntiles_, npairs_, nkb_) : 1;
    nitems = S * ntiles_;
  }
  __device__ __forceinline__ bool next(int& t, int& k0, int& k1, int& split) {
    if (i >= nitems) return false;
    split = i / ntiles;
    t = i - split * ntiles;
    k0 = (int)((int64_t)nkb * split / S);
    k1 = (int)((int64_t)nkb * (split + 1) / S);
    i += npairs;
    return true;
  }
};

// ------------------------------------------------------------------ epilogues
// The forward epilogues write the exp slab straight from registers: each thread holds FC
// consecutive columns of its row as 16-bit values (64 columns: 128 bytes, one whole line)
// and stores them with 32-byte stores. Slab rows past R are skipped (the slab has R rows; rows
// between the chunk's end and R hold values nothing reads, and the zero Xc rows there make
// them finite).
template <typename T>
__device__ __forceinline__ void store_slab(const CallArgs& a, int rr, int col, const uint32_t (&pk)[FC / 2]) {
  if (rr >= (int)a.R) return;
  uint32_t* dst = (uint32_t*)((T*)a.w.slab + (int64_t)rr * a.Vp + col);  // 32-byte aligned
#pragma unroll
  for (int j = 0; j < FC / 16; ++j)
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 8 * j), "r"(pk[8 * j]),
                 "r"(pk[8 * j + 1]), "r"(pk[8 * j + 2]), "r"(pk[8 * j + 3]), "r"(pk[8 * j + 4]),
                 "r"(pk[8 * j + 5]), "r"(pk[8 * j + 6]), "r"(pk[8 * j + 7])
                 : "memory");
}

// r[idx] for a per-thread index 0 <= idx < N by a select tree (indexing the register
// array at run time would move it to local memory).
template <int N>
__device__ __forceinline__ float select_n(const uint32_t (&r)[N], int idx) {
  float x[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) x[i] = __uint_as_float((idx & 1) ? r[2 * i + 1] : r[2 * i]);
#pragma unroll
  for (int w = N / 4, b = 2; w >= 1; w >>= 1, b <<= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) x[i] = (idx & b) ? x[2 * i + 1] : x[2 * i];
  }
  return x[0];
}

// The logit of one accumulator element: acc * ls (+ bias[v]). SCALE: ls != 1 (the
// distillation op's 1/T); BIAS: a bias is added. Rounded multiply and add (no contraction
// into an FMA), so that every place that evaluates a logit gets the same bits.
template <typename T, bool SCALE, bool BIAS>
__device__ __forceinline__ float logit_of(uint32_t acc, int v, float ls, const T* bias) {
  float s = __uint_as_float(acc);
  if (SCALE) s = __fmul_rn(s, ls);
  if (BIAS) s = __fadd_rn(s, to_f<T>(bias[v]));
  return s;
}

// The target logit of a row whose target column lies in the FC columns just loaded
// (loc in [0, FC)). The warp picks it out only when one of its 32 rows has its target
// there (about one 64-column block in 60 at V = 128256), so no per-column comparison runs.
template <typename T, bool SCALE, bool BIAS>
__device__ __forceinline__ void pick_target(const uint32_t (&r)[FC], int loc, int v, float ls, const T* bias,
                                            float& tl) {
  const bool mine = (unsigned)loc < (unsigned)FC;
  if (__any_sync(0xffffffffu, mine)) {
    const float tv = select_n<FC>(r, loc & (FC - 1));
    if (mine) tl = logit_of<T, SCALE, BIAS>(__float_as_uint(tv), v, ls, bias);
  }
}

// The argmax is kept as a value-only maximum per 64 columns (one max instruction per
// logit); the lowest column holding a block's maximum is searched for only when that block
// raises the tile's maximum AND can hold the row's maximum, i.e. its maximum is at least
// the largest tile maximum of the row already written by other tiles of this chunk (thr,
// read from the workspace's running row maxima at the start of the tile). A tile whose
// maximum stays below thr cannot hold the row's argmax: its stored index is never chosen,
// because the merge in finalize takes the index of a tile with the row's largest maximum
// (lowest index among equal maxima), and every such tile searched its own. Most blocks skip
// the search: once a few tiles of a row are done, thr is near the row's maximum.
//
// Lowest column among the 64 just evaluated whose logit equals m (their maximum); s holds
// the logits (columns past the vocabulary hold -inf, never equal to a searched maximum).
__device__ __forceinline__ int find_max_col(const uint32_t (&s)[FC], int vbase, float m) {
  int j0 = 0;
#pragma unroll
  for (int j = FC - 1; j >= 0; --j)
    if (__uint_as_float(s[j]) == m) j0 = j;
  return vbase + j0;
}

// Argmax bookkeeping after a 64-column block of logits s with maximum bm (warp-collective).
__device__ __forceinline__ void argmax_update(const uint32_t (&s)[FC], int vbase, float bm, float thr, float& mx,
                                              int& ai) {
  const bool need = bm > mx && bm >= thr;
  if (__any_sync(0xffffffffu, need)) {
    if (need) ai = find_max_col(s, vbase, bm);
  }
  mx = fmaxf(mx, bm);
}

// 64 columns of the row-reference forward: their maximum (four independent chains), the
// sums of exp(s) (four partial sums) and the packed exp(s) values; the accumulator values
// in r are replaced by the logits (for the argmax search). FULL: every column lies inside
// the vocabulary (all but the last tile), no column test; columns past the vocabulary count
// as -inf (exp 0).
template <typename T, bool FULL, bool SCALE, bool BIAS>
__device__ __forceinline__ void fwd_ref_cols(uint32_t (&r)[FC], int vbase, int V, float ls, const T* bias,
                                             float& bm, float (&sum4)[4], uint32_t (&pk)[FC / 2]) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int jj = 0; jj < FC; jj += 2) {
    const int v = vbase + jj;
    const int u = (jj >> 1) & 3;
    float s0 = -INFINITY, s1 = -INFINITY;
    if (FULL || v < V) s0 = logit_of<T, SCALE, BIAS>(r[jj], v, ls, bias);
    if (FULL || v + 1 < V) s1 = logit_of<T, SCALE, BIAS>(r[jj + 1], v + 1, ls, bias);
    r[jj] = __float_as_uint(s0);
    r[jj + 1] = __float_as_uint(s1);
    m4[u] = fmaxf(m4[u], fmaxf(s0, s1));
    const float e0 = ex2_fast(s0 * LOG2E);
    const float e1 = ex2_fast(s1 * LOG2E);
    sum4[u] += e0 + e1;
    pk[jj / 2] = pack2<T>(e0, e1);
  }
  bm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// The row's running maximum thr (see argmax_update) at the start of a tile.
__device__ __forceinline__ float row_threshold(const CallArgs& a, int rr) {
  if (a.w.rmax == nullptr) return -INFINITY;
  int k;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(k) : "l"(a.w.rmax + rr) : "memory");
  return max_key_value(k);
}

// Per-tile statistics of a row, and its contribution to the running row maximum.
__device__ __forceinline__ void write_tile_stats(const CallArgs& a, int rr, int n, float mx, float sum, int ai,
                                                 float thr, bool want_arg) {
  const int64_t o = (int64_t)rr * a.nvt + n;
  a.w.stm[o] = mx;
  a.w.sts[o] = sum;
  a.w.sti[o] = ai;
  if (want_arg && a.w.rmax != nullptr && mx > thr) atomicMax(a.w.rmax + rr, max_key(mx));
}

// The per-row values a forward epilogue thread needs for a tile: its row within the chunk,
// the row's target (through the compaction index) and the running row maximum. Read before
// the epilogue waits for its accumulator, so that the two dependent global loads and the
// threshold load overlap the wait instead of starting the tile's work.
struct FwdRow {
  int rr;
  bool valid;
  int64_t tg;  // target column of the row (-1: none wanted or not a row of the chunk)
  float thr;
};
__device__ __forceinline__ FwdRow fwd_row(const CallArgs& a, int row0, int rows, int mrow, int q, int lane) {
  FwdRow f;
  f.rr = mrow + q * 32 + lane;
  f.valid = f.rr < rows;
  f.tg = -1;
  f.thr = -INFINITY;
  if (f.valid && a.targets != nullptr) {  // the distillation op needs no argmax
    f.tg = a.targets[a.w.idx[row0 + f.rr]];
    f.thr = row_threshold(a, f.rr);
  }
  return f;
}

// Row-reference forward epilogue: exp(s) needs no tile max, so one pass over TMEM (64
// columns per wait) gives the max / lowest-index argmax, the target logit and the exp
// values, written to the slab.
template <typename T, bool SCALE, bool BIAS>
__device__ __forceinline__ void epilogue_fwd_ref(const CallArgs& a, const FwdRow& fr, int n, uint32_t taddr) {
  const int rr = fr.rr;
  const bool valid = fr.valid;
  const int v0 = n * VT;
  const int V = (int)a.V;
  const bool want_arg = a.targets != nullptr;  // the distillation op needs no argmax
  const float thr = fr.thr;
  // the target's column within this tile, or -1
  const int toff = (fr.tg >= v0 && fr.tg < v0 + BN) ? (int)(fr.tg - v0) : -1;
  const float ls = a.logit_scale;
  const T* bias = (const T*)a.bias;
  const bool full = v0 + BN <= V;
  float mx = -INFINITY, tl = 0.0f;
  float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  int ai = v0;
#pragma unroll 1
  for (int c2 = 0; c2 < BN / FC; ++c2) {
    uint32_t r[FC];
    tmem_ldn<FC>(taddr + c2 * FC, r);
    const int vb = v0 + c2 * FC;
    pick_target<T, SCALE, BIAS>(r, toff - c2 * FC, v0 + toff, ls, bias, tl);
    uint32_t pk[FC / 2];
    float bm;
    if (full) {
      fwd_ref_cols<T, true, SCALE, BIAS>(r, vb, V, ls, bias, bm, sum4, pk);
    } else {
      fwd_ref_cols<T, false, SCALE, BIAS>(r, vb, V, ls, bias, bm, sum4, pk);
    }
    if (want_arg) argmax_update(r, vb, bm, thr, mx, ai);
    if (!want_arg) mx = fmaxf(mx, bm);
    store_slab<T>(a, rr, vb, pk);
  }
  if (valid) {
    write_tile_stats(a, rr, n, mx, (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]), ai, thr, want_arg);
    if (toff >= 0) a.w.tgt[rr] = tl;
  }
}

// Per-tile forward epilogue, first pass over 64 columns: their maximum (four chains); the
// accumulator values in r are replaced by the logits (-inf past the vocabulary).
template <typename T, bool FULL, bool SCALE, bool BIAS>
__device__ __forceinline__ float fwd_tile_max(uint32_t (&r)[FC], int vbase, int V, float ls, const T* bias) {
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < FC; ++j) {
    const int v = vbase + j;
    const float s = (FULL || v < V) ? logit_of<T, SCALE, BIAS>(r[j], v, ls, bias) : -INFINITY;
    r[j] = __float_as_uint(s);
    m4[j & 3] = fmaxf(m4[j & 3], s);
  }
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// Per-tile forward epilogue, second pass over 64 columns: exp(s - max) (base 2, mxl =
// max * log2 e) packed for the slab, and their sums (four partial sums).
template <typename T, bool FULL, bool SCALE, bool BIAS>
__device__ __forceinline__ void fwd_tile_exp(const uint32_t (&r)[FC], int vbase, int V, float ls, const T* bias,
                                             float mxl, float (&sum4)[4], uint32_t (&pk)[FC / 2]) {
#pragma unroll
  for (int j = 0; j < FC; j += 2) {
    const int v = vbase + j;
    float e0 = 0.0f, e1 = 0.0f;
    if (FULL || v < V) e0 = ex2_fast(fmaf(logit_of<T, SCALE, BIAS>(r[j], v, ls, bias), LOG2E, -mxl));
    if (FULL || v + 1 < V) e1 = ex2_fast(fmaf(logit_of<T, SCALE, BIAS>(r[j + 1], v + 1, ls, bias), LOG2E, -mxl));
    sum4[(j >> 1) & 3] += e0 + e1;
    pk[j / 2] = pack2<T>(e0, e1);
  }
}

// Per-tile forward epilogue (fp16 inputs, dbias, the distillation op, a chunk outside the
// row-reference window): a first pass over TMEM for the max / argmax / target logit, a
// second for exp(s - max) into the slab.
template <typename T, bool SCALE, bool BIAS>
__device__ __forceinline__ void epilogue_fwd(const CallArgs& a, const FwdRow& fr, int n, uint32_t taddr) {
  const int rr = fr.rr;
  const bool valid = fr.valid;
  const int v0 = n * VT;
  const int V = (int)a.V;
  const bool want_arg = a.targets != nullptr;
  const float thr = fr.thr;
  const int toff = (fr.tg >= v0 && fr.tg < v0 + BN) ? (int)(fr.tg - v0) : -1;
  const float ls = a.logit_scale;
  const T* bias = (const T*)a.bias;
  const bool full = v0 + BN <= V;
  float mx = -INFINITY, tl = 0.0f;
  int ai = v0;
#pragma unroll 1
  for (int c2 = 0; c2 < BN / FC; ++c2) {
    uint32_t r[FC];
    tmem_ldn<FC>(taddr + c2 * FC, r);
    const int vb = v0 + c2 * FC;
    pick_target<T, SCALE, BIAS>(r, toff - c2 * FC, v0 + toff, ls, bias, tl);
    const float bm = full ? fwd_tile_max<T, true, SCALE, BIAS>(r, vb, V, ls, bias)
                          : fwd_tile_max<T, false, SCALE, BIAS>(r, vb, V, ls, bias);
    if (want_arg) argmax_update(r, vb, bm, thr, mx, ai);
    else mx = fmaxf(mx, bm);
  }
  // exp(s - max) to the slab, 64 columns at a time
  float sum4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const float mxl = a.ref_mode ? 0.0f : mx * LOG2E;  // row-reference mode stores exp(s)
#pragma unroll 1
  for (int c2 = 0; c2 < BN / FC; ++c2) {
    uint32_t r[FC];
    tmem_ldn<FC>(taddr + c2 * FC, r);
    uint32_t pk[FC / 2];
    const int vb = v0 + c2 * FC;
    if (full) fwd_tile_exp<T, true, SCALE, BIAS>(r, vb, V, ls, bias, mxl, sum4, pk);
    else fwd_tile_exp<T, false, SCALE, BIAS>(r, vb, V, ls, bias, mxl, sum4, pk);
    store_slab<T>(a, rr, vb, pk);
  }
  if (valid) {
    write_tile_stats(a, rr, n, mx, (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]), ai, thr, want_arg);
    if (toff >= 0) a.w.tgt[rr] = tl;
  }
}

// Dispatch of the forward epilogues on the logit scale and the bias (warp-uniform).
template <typename T, bool SCALE, bool BIAS>
__device__ __forceinline__ void epilogue_fwd_any3(const CallArgs& a, const FwdRow& fr, int n, uint32_t taddr) {
  if (a.ref_mode) epilogue_fwd_ref<T, SCALE, BIAS>(a, fr, n, taddr);
  else epilogue_fwd<T, SCALE, BIAS>(a, fr, n, taddr);
}
// GEN: 0 for launches with no bias and a logit scale of 1 (the cross-entropy op without
// bias), 1 with a bias and a scale of 1, 2 with another scale (the distillation op at
// T != 1). Each is a kernel build of its own, so that the common ones keep all their values
// in registers.
template <typename T, int GEN>
__device__ __forceinline__ void epilogue_fwd_any(const CallArgs& a, const FwdRow& fr, int n, uint32_t taddr) {
  if constexpr (GEN == 0) {
    epilogue_fwd_any3<T, false, false>(a, fr, n, taddr);
  } else if constexpr (GEN == 1) {
    epilogue_fwd_any3<T, false, true>(a, fr, n, taddr);
  } else {
    if (a.bias != nullptr) epilogue_fwd_any3<T, true, true>(a, fr, n, taddr);
    else epilogue_fwd_any3<T, true, false>(a, fr, n, taddr);
  }
}

// dst tile += cbar * acc through TMA reduce-add (dst = dW for DW; for DX the fp32
// accumulator buffer starting at row yoff; in row-reference mode each dX row is also
// scaled by its rsc). Each epilogue warp owns 32 rows (its TMEM lane quadrant) and stages
// 32 columns at a time (32 x 128 B, 128-byte swizzle: 16-byte chunk j of row r sits at
// chunk j ^ (r % 8)) in NBUF rotating buffers; the TMA unit adds the box into dst in L2.
// A dW element gets exactly one add per launch (one owning pair); a dX buffer element at
// most two (K splits), added to zero: either way the result does not depend on timing.
// Boxes past the destination's extent are clipped by the TMA unit.
//
// HALF (the eight-warp epilogue of the wide tiles, 4 KB of staging per warp, and every
// 16-bit destination): two 2 KB buffers of 32 rows x 64 bytes (64-byte swizzle: 16-byte
// chunk j of row r at chunk j ^ ((r / 2) % 4)), so that a warp stages the next box while
// the TMA unit still reads the previous one. A box is 16 fp32 columns, or 32 columns of a
// 16-bit destination D (same-dtype dW: the L2 adds in D), the map's box accordingly
// {16, 32} or {32, 32}. STORE: the box overwrites dst instead of adding to it (the first
// chunk of a call with FLCE_FLAG_DW_OVERWRITE).
template <int NBUF, bool HALF, typename D, int HB>
__device__ __forceinline__ void epilogue_reduce(const CallArgs& a, const CUtensorMap* tmC, uint8_t* stg,
                                                int mrow, int n, int ylimit, int yoff, uint32_t taddr,
                                                int q, int lane, float cb, const float* rsc, bool store,
                                                uint32_t& epi_it) {
  const int H = (int)a.H;
  const int y = mrow + q * 32;
  if (y >= ylimit) return;  // this warp's 32 rows lie past the destination (warp-uniform)
  if (rsc != nullptr) cb *= rsc[y + lane];  // y + lane < ylimit = R (multiples of 32)
  constexpr bool F32 = std::is_same<D, float>::value;
  if (HALF || !F32) {
    constexpr int BOX = F32 ? 16 : 32;  // columns per 64-byte box row
#pragma unroll 1
    for (int cc = 0; cc < BN / 32; ++cc) {
      const int x = n * BN + cc * 32;
      if (x >= H) break;  // warp-uniform
      uint32_t r[32];
      tmem_ld32(taddr + cc * 32, r);
#pragma unroll
      for (int h = 0; h < 32 / BOX; ++h) {
        if (x + BOX * h >= H) break;  // warp-uniform
        uint8_t* buf = stg + (epi_it % HB) * (EPI_BUF_BYTES / 2);
        if (lane == 0) bulk_wait_read<HB - 1>();  // the op that last read this buffer is done
        __syncwarp();
        uint8_t* row = buf + lane * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 v;
          if constexpr (F32) {
            const int c = 16 * h + 4 * j;
            v = make_uint4(__float_as_uint(cb * __uint_as_float(r[c + 0])),
                           __float_as_uint(cb * __uint_as_float(r[c + 1])),
                           __float_as_uint(cb * __uint_as_float(r[c + 2])),
                           __float_as_uint(cb * __uint_as_float(r[c + 3])));
          } else {
            const int c = 8 * j;
            v = make_uint4(pack2<D>(cb * __uint_as_float(r[c + 0]), cb * __uint_as_float(r[c + 1])),
                           pack2<D>(cb * __uint_as_float(r[c + 2]), cb * __uint_as_float(r[c + 3])),
                           pack2<D>(cb * __uint_as_float(r[c + 4]), cb * __uint_as_float(r[c + 5])),
                           pack2<D>(cb * __uint_as_float(r[c + 6]), cb * __uint_as_float(r[c + 7])));
          }
          *(uint4*)(row + ((j ^ ((lane >> 1) & 3)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (store) tma_store_2d(tmC, smem_u32(buf), x + BOX * h, y + yoff);
          else tma_reduce_add_2d(tmC, smem_u32(buf), x + BOX * h, y + yoff);
          bulk_commit();
        }
        ++epi_it;
      }
    }
    return;
  }
#pragma unroll 1
  for (int cc = 0; cc < BN / 32; ++cc) {
    const int x = n * BN + cc * 32;
    if (x >= H) break;  // warp-uniform
    uint32_t r[32];
    tmem_ld32(taddr + cc * 32, r);
    uint8_t* buf = stg + (epi_it % NBUF) * EPI_BUF_BYTES;
    if (lane == 0) bulk_wait_read<NBUF - 1>();  // the reduce that last read this buffer is done
    __syncwarp();
    uint8_t* row = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float4 v = make_float4(cb * __uint_as_float(r[4 * j + 0]), cb * __uint_as_float(r[4 * j + 1]),
                             cb * __uint_as_float(r[4 * j + 2]), cb * __uint_as_float(r[4 * j + 3]));
      *(float4*)(row + ((j ^ (lane & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (store) tma_store_2d(tmC, smem_u32(buf), x, y + yoff);
      else tma_reduce_add_2d(tmC, smem_u32(buf), x, y + yoff);
      bulk_commit();
    }
    ++epi_it;
  }
}

// ------------------------------------------------------------------ the kernel
template <int MODE, typename T, int NB, int GEN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CallArgs a,
              const int chunk) {
  constexpr int STAGES = stages_of<NB>();
  constexpr int SBYTES = stage_bytes<NB>();
  constexpr int NACC = nacc_of<NB>();
  constexpr int NEPI = epi_warps_of<NB>();
  constexpr int NBUF = epi_nbuf_of<NB>();
  if (a.run_if != nullptr && *a.run_if == 0) return;  // both CTAs of a pair read the same word
  int row0 = 0, rows = 0;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const TileSpace ts = tile_space<MODE, NB>(a, rows);
  const int ntiles = ts.mt * ts.nt;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), npairs = (int)nclusters_x();
  // both CTAs of a pair take the same decision
  if (ts.nkb <= 0 || pair >= Items<MODE>(0, npairs, ntiles, ts.nkb).nitems) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* epi_stage = smem + STAGES * SBYTES;
  uint64_t* bars = (uint64_t*)(smem + STAGES * SBYTES + epi_bytes_m<MODE, NB>());
  uint32_t* tmem_slot = (uint32_t*)(bars + NUM_BARS);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* copies = (int*)(tmem_slot + 2);  // per stage: phases this CTA's producer filled / armed
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  auto tempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 + s); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, mapa(smem_u32((const void*)abort_flag), rank ^ 1u), a.w.status, a.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // leader: one arrive (its expect_tx for both halves)
      mbar_init(empty_bar(s), 1);  // one MMA commit per phase (multicast to both CTAs)
      copies[s] = 0;
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(tfull_bar(s), 1);             // one MMA commit per tile (multicast)
      mbar_init(tempty_bar(s), 2 * NEPI);     // leader: local + peer epilogue warps
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmA) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmB) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int s = 0;
      uint32_t ph = 0;
      const bool stall = (a.flags & FLCE_FLAG_DEBUG_STALL) && MODE == FWD && leader;
      const int half = (int)rank * BM;  // this CTA's 128-row half of A and of each B sub-tile
      Items<MODE> items(pair, npairs, ntiles, ts.nkb);
      int tile, k0, k1, split;
      bool first = true;
      while (items.next(tile, k0, k1, split)) {
        int m, n;
        tile_coords<MODE>(ts, tile, m, n);
        int kb = k0;
        for (; kb < k1; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, ab, true)) break;
          const uint32_t fb = leader ? full_bar(s) : mapa(full_bar(s), 0);
          if (leader) mbar_expect_tx(full_bar(s), 2 * SBYTES);
          if (!(stall && first && kb == k1 - 1)) {
            const uint32_t adst = smem_u32(smem + s * SBYTES);
            const uint32_t bdst = adst + A_BYTES;
            if (MODE == FWD) {
              tma_load_2d(adst, &tmA, fb, kb * BK, m * 2 * BM + half);
#pragma unroll
              for (int j = 0; j < NB; ++j)
                tma_load_2d(bdst + j * B_BYTES, &tmB, fb, kb * BK, (n * NB + j) * BN + half);
            } else if (MODE == DX) {
              tma_load_2d(adst, &tmA, fb, kb * BK, m * 2 * BM + half);
#pragma unroll
              for (int j = 0; j < NB; ++j)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                  tma_load_2d(bdst + j * B_BYTES + jj * BOX_BYTES, &tmB, fb,
                              (n * NB + j) * BN + half + jj * 64, kb * BK);
            } else {
#pragma unroll
              for (int jj = 0; jj < 2; ++jj)
                tma_load_2d(adst + jj * BOX_BYTES, &tmA, fb, m * 2 * BM + half + jj * 64, kb * BK);
#pragma unroll
              for (int j = 0; j < NB; ++j)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                  tma_load_2d(bdst + j * B_BYTES + jj * BOX_BYTES, &tmB, fb,
                              (n * NB + j) * BN + half + jj * 64, kb * BK);
            }
          }
          copies[s] += 1;  // leader: phases armed; peer: phases filled
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (kb < k1) break;
        first = false;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader CTA)
      constexpr uint32_t idesc = make_idesc<MODE, T>();
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      Items<MODE> items(pair, npairs, ntiles, ts.nkb);
      int tile, k0, k1, split;
      for (; ok && items.next(tile, k0, k1, split); ++it) {
        const int as = it % NACC;
        const uint32_t aph = (uint32_t)(it / NACC) & 1u;
        if (!wait_bounded(tempty_bar(as), aph ^ 1u, ab, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(as * NB * BN);
        for (int kb = k0; kb < k1; ++kb) {
          if (!wait_bounded(full_bar(s), ph, ab, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t abase = smem_u32(smem + s * SBYTES);
          const uint32_t bbase = abase + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = MODE == DW ? sdesc(abase + k * 2048, 8192, 1024) : sdesc(abase + k * 32, 16, 1024);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const uint32_t bj = bbase + j * B_BYTES;
              const uint64_t bd = MODE == FWD ? sdesc(bj + k * 32, 16, 1024) : sdesc(bj + k * 2048, 8192, 1024);
              mma_f16(d + (uint32_t)(j * BN), ad, bd, idesc, (kb != k0 || k != 0) ? 1u : 0u);
            }
          }
          mma_commit_pair(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull_bar(as));
      }
      // every MMA issued completes before TMEM is freed or shared memory released
      mma_commit_local(drain_bar);
      wait_bounded(drain_bar, 0u, ab, false);
    }
  } else if (warp - 2 < NEPI) {
    // ---------------- epilogue warps (both CTAs): warp w reads TMEM lane quadrant w % 4
    // of sub-tile (w - 2) / 4
    const int q = warp & 3;
    const int j = (warp - 2) >> 2;
    const float cb = MODE == FWD ? 0.0f : a.w.ctrl->cbar;
    const float* rsc = (MODE == DX && a.ref_mode && a.w.ctrl->fb == 0) ? a.w.rsc : nullptr;
    // dW overwrite: the first chunk of the call stores its tiles, later chunks add
    const bool ovw = MODE == DW && (a.flags & FLCE_FLAG_DW_OVERWRITE) && chunk == 0;
    uint8_t* stg = epi_stage + (warp - 2) * epi_warp_bytes_of<NB>();
    uint32_t epi_it = 0;
    int it = 0;
    Items<MODE> items(pair, npairs, ntiles, ts.nkb);
    int tile, k0, k1, split;
    for (; items.next(tile, k0, k1, split); ++it) {
      const int as = it % NACC;
      const uint32_t aph = (uint32_t)(it / NACC) & 1u;
      int m, n;
      tile_coords<MODE>(ts, tile, m, n);
      const int nsub = n * NB + j;  // this warp's 256-column sub-tile of the output
      const int mrow = m * 2 * BM + (int)rank * BM;
      FwdRow fr;
      if (MODE == FWD) fr = fwd_row(a, row0, rows, mrow, q, lane);  // loads overlap the wait
      bool ok = wait_bounded(tfull_bar(as), aph, ab, true);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((as * NB + j) * BN);
      if (nsub < ts.nsub) {
        if (MODE == FWD)
          epilogue_fwd_any<T, GEN>(a, fr, nsub, taddr);
        else if (MODE == DW && a.dW_dt != FLCE_F32)
          epilogue_reduce<NBUF, (NB == 2), T, half_bufs_of<NB>()>(a, &tmC, stg, mrow, nsub, (int)a.V, 0, taddr, q, lane, cb,
                                              nullptr, ovw, epi_it);
        else
          epilogue_reduce<NBUF, (NB == 2), float, half_bufs_of<NB>()>(a, &tmC, stg, mrow, nsub, MODE == DX ? (int)a.R : (int)a.V,
                                                  MODE == DX ? (split >> 1) * (int)a.R : 0, taddr, q, lane,
                                                  cb, rsc, MODE == DW && ovw, epi_it);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(as));
        else mbar_arrive_cluster(mapa(tempty_bar(as), 0));
      }
    }
    // every store / reduce this warp issued has finished reading its staging buffer and
    // written its destination
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ---------------- teardown
  tc_fence_before();
  cluster_sync();  // no role of either CTA issues anything after this point
  if (warp == 0 && lane == 0 && leader) {
    // Every copy either CTA issued must land before the pair frees its shared memory. The
    // peer's copies complete on the leader's barriers; an aborted pipeline can leave the
    // two producers one phase apart on a stage, which is reconciled here.
    for (int s = 0; s < STAGES; ++s) {
      const int mine = copies[s];
      const int peer = (int)ld_cluster_u32(mapa(smem_u32(&copies[s]), 1));
      int last = mine;
      if (peer > mine) {
        mbar_expect_tx(full_bar(s), SBYTES);  // arm the phase only the peer filled
        last = peer;
      } else if (peer < mine) {
        mbar_complete_tx(full_bar(s), SBYTES);  // the peer's half never came
      }
      if (last > 0) wait_bounded(full_bar(s), (uint32_t)(last - 1) & 1u, ab, false);
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ merged dX + dW launch
// One persistent launch runs a chunk's dX items (256 x 512 tiles over K = V, split in up to
// four K ranges as in the DX mode) and its dW tiles (256 x 512 over K = chunk rows). The
// pairs take items from a device-wide queue, an atomic counter in the workspace's control
// record, in index order: item g < n_dx is dX item g (split-major), item g >= n_dx the dW
// tile g - n_dx. A pair that finishes its last dX item starts on dW tiles at once instead of
// idling through dX's last partial wave, and the dW tiles in flight still walk the slab in
// step. The leader CTA's producer draws each index and hands it to the other roles of both
// CTAs through a ring of QD slots in shared memory (full / empty barriers per slot). Results
// do not depend on which pair runs which item: a dX buffer element still receives at most two
// adds onto zero, and each dW tile is added by the one pair that drew it.
constexpr int QD = 4;
constexpr int Q_CONSUMERS = 2 + 2 * 8;  // peer producer, MMA issuer, both CTAs' epilogue warps
constexpr int NUM_BARS_BWD = NUM_BARS + 2 * QD;

struct BwdSpace {
  TileSpace dx, dw;
  int S, ntx, n_dx, n_items;
};
__device__ __forceinline__ BwdSpace bwd_space(const CallArgs& a, int rows, int npairs) {
  BwdSpace b;
  b.dx = tile_space<DX, 2>(a, rows);
  b.dw = tile_space<DW, 2>(a, rows);
  b.ntx = b.dx.mt * b.dx.nt;
#if defined(FLCE_BWD_DX_SPLITS) && FLCE_BWD_DX_SPLITS > 0
  static_assert(FLCE_BWD_DX_SPLITS <= DX_MAX_SPLITS, "two dX buffers take at most four splits");
  b.S = FLCE_BWD_DX_SPLITS < b.dx.nkb ? FLCE_BWD_DX_SPLITS : b.dx.nkb;
#else
  b.S = dx_splits(b.ntx, npairs, b.dx.nkb);
#endif
  b.n_dx = b.S * b.ntx;
  b.n_items = b.n_dx + b.dw.mt * b.dw.nt;
  return b;
}
struct BwdItem {
  int dw, m, n, k0, k1, split;
};
__device__ __forceinline__ BwdItem bwd_item(const BwdSpace& b, int g) {
  BwdItem it;
  if (g < b.n_dx) {
    it.dw = 0;
    it.split = g / b.ntx;
    const int t = g - it.split * b.ntx;
    it.n = t % b.dx.nt;  // n fastest: the pairs in flight share the slab rows
    it.m = t / b.dx.nt;
    it.k0 = (int)((int64_t)b.dx.nkb * it.split / b.S);
    it.k1 = (int)((int64_t)b.dx.nkb * (it.split + 1) / b.S);
  } else {
    const int t = g - b.n_dx;
    it.dw = 1;
    it.split = 0;
    it.n = t % b.dw.nt;  // n fastest: the pairs in flight share the slab columns
    it.m = t / b.dw.nt;
    it.k0 = 0;
    it.k1 = b.dw.nkb;
  }
  return it;
}

// Bounded wait with cluster-scope acquire, for barriers that another CTA's release-arrive
// completes together with data it stored into this CTA's shared memory (the queue slots).
__device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const Abort& ab) {
  const uint64_t t0 = gtimer();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(50000u)
        : "memory");
    if (ok) return true;
    if (*ab.flag) return false;
    if (gtimer() - t0 > ab.timeout_ns) {
      *ab.flag = 1;
      st_cluster_u32(ab.peer_flag, 1u);
      atomicOr(ab.status, ST_TIMEOUT);
      return false;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_bwd(const __grid_constant__ CUtensorMap tmAx, const __grid_constant__ CUtensorMap tmBx,
               const __grid_constant__ CUtensorMap tmCx, const __grid_constant__ CUtensorMap tmAw,
               const __grid_constant__ CUtensorMap tmBw, const __grid_constant__ CUtensorMap tmCw,
               const __grid_constant__ CallArgs a, const int chunk) {
  constexpr int NB = 2;
  constexpr int STAGES = stages_of<NB>();
  constexpr int SBYTES = stage_bytes<NB>();
  constexpr int NEPI = epi_warps_of<NB>();
  constexpr int NBUF = epi_nbuf_of<NB>();
  constexpr int HB = half_bufs_of<NB>();
  int row0 = 0, rows = 0;
  if (!chunk_bounds(a.w.ctrl, chunk, row0, rows)) return;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), npairs = (int)nclusters_x();
  const BwdSpace bs = bwd_space(a, rows, npairs);
  // both CTAs of a pair take the same decision; pairs beyond the item count never draw
  if (bs.dx.nkb <= 0 || bs.dw.nkb <= 0 || pair >= bs.n_items) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* epi_stage = smem + STAGES * SBYTES;
  uint64_t* bars = (uint64_t*)(smem + STAGES * SBYTES + epi_bytes_of<NB>());
  uint32_t* tmem_slot = (uint32_t*)(bars + NUM_BARS_BWD);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* copies = (int*)(tmem_slot + 2);  // per stage: phases this CTA's producer filled / armed
  int* qitem = copies + STAGES;         // the queue ring: item index per slot
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t tfull = bar0 + 8u * (2 * STAGES);
  const uint32_t tempty = bar0 + 8u * (2 * STAGES + 2);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto qfull_bar = [&](int q) { return bar0 + 8u * (NUM_BARS + q); };
  auto qempty_bar = [&](int q) { return bar0 + 8u * (NUM_BARS + QD + q); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, mapa(smem_u32((const void*)abort_flag), rank ^ 1u), a.w.status, a.timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      copies[s] = 0;
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * NEPI);
    mbar_init(drain_bar, 1);
    for (int q = 0; q < QD; ++q) {
      mbar_init(qfull_bar(q), 1);              // the leader's producer, locally or remotely
      mbar_init(qempty_bar(q), Q_CONSUMERS);   // used in the leader CTA
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmAx) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmBx) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmAw) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmBw) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Next item of this pair from the queue ring (every role but the drawing one): false on
  // abort. The slot is released on the leader's empty barrier once the index is read.
  auto take = [&](int& slot, uint32_t& qph, int& g) -> bool {
    if (!wait_bounded_cluster(qfull_bar(slot), qph, ab)) return false;
    g = ((volatile int*)qitem)[slot];
    return true;
  };
  auto release_slot = [&](int slot) {
    if (leader) mbar_arrive(qempty_bar(slot));
    else mbar_arrive_cluster(mapa(qempty_bar(slot), 0));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs); the leader's also draws the items
      int s = 0;
      uint32_t ph = 0;
      const int half = (int)rank * BM;
      int slot = 0;
      uint32_t qph = 0;
      const bool stall = (a.flags & FLCE_FLAG_DEBUG_STALL_BWD) && leader;
      bool first = true;
      for (;;) {
        int g;
        if (leader) {
          // the slot's previous index has been read by every role of both CTAs
          if (!wait_bounded_cluster(qempty_bar(slot), qph ^ 1u, ab)) break;
          g = atomicAdd(&a.w.ctrl->queue, 1);
          qitem[slot] = g;
          st_cluster_u32(mapa(smem_u32(&qitem[slot]), 1), (uint32_t)g);
          mbar_arrive(qfull_bar(slot));
          mbar_arrive_cluster(mapa(qfull_bar(slot), 1));
        } else {
          if (!take(slot, qph, g)) break;
          release_slot(slot);
        }
        if (++slot == QD) {
          slot = 0;
          qph ^= 1u;
        }
        if (g >= bs.n_items) break;
        const BwdItem it = bwd_item(bs, g);
        int kb = it.k0;
        for (; kb < it.k1; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, ab, true)) break;
          const uint32_t fb = leader ? full_bar(s) : mapa(full_bar(s), 0);
          if (leader) mbar_expect_tx(full_bar(s), 2 * SBYTES);
          const uint32_t adst = smem_u32(smem + s * SBYTES);
          const uint32_t bdst = adst + A_BYTES;
          if (stall && first && kb == it.k1 - 1) {
            // testing only: this stage is armed but never filled
          } else if (it.dw) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
              tma_load_2d(adst + jj * BOX_BYTES, &tmAw, fb, it.m * 2 * BM + half + jj * 64, kb * BK);
#pragma unroll
            for (int j = 0; j < NB; ++j)
#pragma unroll
              for (int jj = 0; jj < 2; ++jj)
                tma_load_2d(bdst + j * B_BYTES + jj * BOX_BYTES, &tmBw, fb,
                            (it.n * NB + j) * BN + half + jj * 64, kb * BK);
          } else {
            tma_load_2d(adst, &tmAx, fb, kb * BK, it.m * 2 * BM + half);
#pragma unroll
            for (int j = 0; j < NB; ++j)
#pragma unroll
              for (int jj = 0; jj < 2; ++jj)
                tma_load_2d(bdst + j * B_BYTES + jj * BOX_BYTES, &tmBx, fb,
                            (it.n * NB + j) * BN + half + jj * 64, kb * BK);
          }
          copies[s] += 1;  // leader: phases armed; peer: phases filled
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (kb < it.k1) break;
        first = false;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader CTA)
      constexpr uint32_t idesc_dx = make_idesc<DX, T>();
      constexpr uint32_t idesc_dw = make_idesc<DW, T>();
      int s = 0;
      uint32_t ph = 0;
      int slot = 0;
      uint32_t qph = 0;
      bool ok = true;
      for (int n_it = 0; ok; ++n_it) {
        int g;
        if (!take(slot, qph, g)) break;
        release_slot(slot);
        if (++slot == QD) {
          slot = 0;
          qph ^= 1u;
        }
        if (g >= bs.n_items) break;
        const BwdItem it = bwd_item(bs, g);
        if (!wait_bounded(tempty, ((uint32_t)n_it & 1u) ^ 1u, ab, true)) break;
        tc_fence_after();
        const uint32_t idesc = it.dw ? idesc_dw : idesc_dx;
        for (int kb = it.k0; kb < it.k1; ++kb) {
          if (!wait_bounded(full_bar(s), ph, ab, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t abase = smem_u32(smem + s * SBYTES);
          const uint32_t bbase = abase + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // dX: A = slab K-major; dW: A = slab^T MN-major; B MN-major for both
            const uint64_t ad = it.dw ? sdesc(abase + k * 2048, 8192, 1024) : sdesc(abase + k * 32, 16, 1024);
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const uint64_t bd = sdesc(bbase + j * B_BYTES + k * 2048, 8192, 1024);
              mma_f16(tmem_base + (uint32_t)(j * BN), ad, bd, idesc, (kb != it.k0 || k != 0) ? 1u : 0u);
            }
          }
          mma_commit_pair(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(tfull);
      }
      mma_commit_local(drain_bar);
      wait_bounded(drain_bar, 0u, ab, false);
    }
  } else if (warp - 2 < NEPI) {
    // ---------------- epilogue warps (both CTAs): TMEM lane quadrant warp % 4 of 256-column
    // sub-tile (warp - 2) / 4
    const int q = warp & 3;
    const int j = (warp - 2) >> 2;
    const float cb = a.w.ctrl->cbar;
    const float* rsc = (a.ref_mode && a.w.ctrl->fb == 0) ? a.w.rsc : nullptr;
    const bool ovw = (a.flags & FLCE_FLAG_DW_OVERWRITE) && chunk == 0;
    uint8_t* stg = epi_stage + (warp - 2) * epi_warp_bytes_of<NB>();
    uint32_t epi_it = 0;
    int slot = 0;
    uint32_t qph = 0;
    for (int n_it = 0;; ++n_it) {
      int g;
      bool ok = take(slot, qph, g);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) release_slot(slot);
      if (++slot == QD) {
        slot = 0;
        qph ^= 1u;
      }
      if (g >= bs.n_items) break;
      const BwdItem it = bwd_item(bs, g);
      ok = wait_bounded(tfull, (uint32_t)n_it & 1u, ab, true);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int nsub = it.n * NB + j;
      const int mrow = it.m * 2 * BM + (int)rank * BM;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(j * BN);
      if (nsub < bs.dx.nsub) {
        if (!it.dw)
          epilogue_reduce<NBUF, true, float, HB>(a, &tmCx, stg, mrow, nsub, (int)a.R, (it.split >> 1) * (int)a.R,
                                                 taddr, q, lane, cb, rsc, false, epi_it);
        else if (a.dW_dt != FLCE_F32)
          epilogue_reduce<NBUF, true, T, HB>(a, &tmCw, stg, mrow, nsub, (int)a.V, 0, taddr, q, lane, cb, nullptr, ovw,
                                             epi_it);
        else
          epilogue_reduce<NBUF, true, float, HB>(a, &tmCw, stg, mrow, nsub, (int)a.V, 0, taddr, q, lane, cb, nullptr,
                                                 ovw, epi_it);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty);
        else mbar_arrive_cluster(mapa(tempty, 0));
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // ---------------- teardown (as in k_gemm_tc)
  tc_fence_before();
  cluster_sync();
  if (warp == 0 && lane == 0 && leader) {
    for (int s = 0; s < STAGES; ++s) {
      const int mine = copies[s];
      const int peer = (int)ld_cluster_u32(mapa(smem_u32(&copies[s]), 1));
      int last = mine;
      if (peer > mine) {
        mbar_expect_tx(full_bar(s), SBYTES);
        last = peer;
      } else if (peer < mine) {
        mbar_complete_tx(full_bar(s), SBYTES);
      }
      if (last > 0) wait_bounded(full_bar(s), (uint32_t)(last - 1) & 1u, ab, false);
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// 2-D tiled map over a row-major matrix [outer, inner] with row pitch `pitch_bytes`;
// 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* m, const void* ptr, int dt, uint64_t inner, uint64_t outer,
              uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const CUtensorMapDataType ty = dt == FLCE_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dt == FLCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, ty, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch as clusters of 2 CTAs, one pair per pair tile up to the number of pairs that fit
// the GPU at once (persistent).
template <int MODE, typename T, int NB, int GEN>
cudaError_t launch_t(const CallArgs& a, int chunk, cudaStream_t s, const CUtensorMap& A,
                     const CUtensorMap& B, const CUtensorMap& C, int64_t pair_tiles_max) {
  auto kern = k_gemm_tc<MODE, T, NB, GEN>;
  constexpr int smem = smem_bytes<MODE, NB>();
  // per-device cache of the pairs that fit at once (the shared-memory attribute is set on
  // the first launch of each device); concurrent first launches may both set and store it
  static std::atomic<int> max_pairs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dev < 0 || dev >= 64 || max_pairs[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (unsigned)(num_sms() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) max_pairs[dev].store(n, std::memory_order_relaxed);
    else return cudaErrorInvalidDevice;
  }
  // (the shared-memory attribute, set once per device above, persists: later launches,
  // including ones captured into a CUDA graph, enqueue the kernel only)
  const int mp = max_pairs[dev].load(std::memory_order_relaxed);
  const int64_t pairs = pair_tiles_max < mp ? pair_tiles_max : mp;
  if (pairs <= 0) return cudaSuccess;
  cfg.gridDim = dim3(2 * (unsigned)pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, A, B, C, a, chunk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MODE, int NB>
cudaError_t launch_mode(const CallArgs& a, int chunk, cudaStream_t s, const CUtensorMap& A,
                        const CUtensorMap& B, const CUtensorMap& C, int64_t tiles_max) {
  // the forward has builds of its own for launches with a bias or a logit scale
  if constexpr (MODE == FWD) {
    if (a.logit_scale != 1.0f) {
      if (a.dt == FLCE_BF16) return launch_t<MODE, __nv_bfloat16, NB, 2>(a, chunk, s, A, B, C, tiles_max);
      return launch_t<MODE, __half, NB, 2>(a, chunk, s, A, B, C, tiles_max);
    }
    if (a.bias != nullptr) {
      if (a.dt == FLCE_BF16) return launch_t<MODE, __nv_bfloat16, NB, 1>(a, chunk, s, A, B, C, tiles_max);
      return launch_t<MODE, __half, NB, 1>(a, chunk, s, A, B, C, tiles_max);
    }
  }
  if (a.dt == FLCE_BF16) return launch_t<MODE, __nv_bfloat16, NB, 0>(a, chunk, s, A, B, C, tiles_max);
  return launch_t<MODE, __half, NB, 0>(a, chunk, s, A, B, C, tiles_max);
}

}  // namespace tc

bool tc_supported(const CallArgs& a) {
  if (a.dt != FLCE_BF16 && a.dt != FLCE_F16) return false;
  if (a.H % 8 != 0) return false;  // TMA: the W row pitch must be a multiple of 16 bytes
  if (a.H > (1LL << 30) || a.V > (1LL << 30)) return false;
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_fwd_tc(const CallArgs& a, int chunk, cudaStream_t s) {
  CUtensorMap A, B;
  const uint64_t esz = 2;
  if (!tc::make_map(&A, a.w.xc, a.dt, a.H, a.R, a.Hp * esz, 64, 128)) return cudaErrorInvalidValue;
  if (!tc::make_map(&B, a.W, a.dt, a.H, a.V, a.H * esz, 64, 128)) return cudaErrorInvalidValue;
  const int64_t mt = (a.R + 255) / 256;
  // the forward epilogue writes the slab with plain stores: the third map is not read
  if (a.H >= FWD_WIDE_MIN_H) return tc::launch_mode<tc::FWD, 2>(a, chunk, s, A, B, B, mt * ((a.nvt + 1) / 2));
  return tc::launch_mode<tc::FWD, 1>(a, chunk, s, A, B, B, mt * a.nvt);
}

cudaError_t launch_dx_tc(const CallArgs& a, int chunk, cudaStream_t s) {
  CUtensorMap A, B;
  const uint64_t esz = 2;
  if (!tc::make_map(&A, a.w.slab, a.dt, a.V, a.R, a.Vp * esz, 64, 128)) return cudaErrorInvalidValue;
  if (!tc::make_map(&B, a.W, a.dt, a.H, a.V, a.H * esz, 64, 64)) return cudaErrorInvalidValue;
  CUtensorMap C;  // the two fp32 accumulator buffers [2R, H] (K splits 0-1 and 2-3)
  if (!tc::make_map(&C, a.w.dxacc, FLCE_F32, a.H, 2 * a.R, a.H * 4, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const int64_t tiles = tc::DX_MAX_SPLITS * ((a.R + 255) / 256) * (((a.H + 255) / 256 + 1) / 2);
  return tc::launch_mode<tc::DX, 2>(a, chunk, s, A, B, C, tiles);
}

cudaError_t launch_dw_tc(const CallArgs& a, int chunk, cudaStream_t s) {
  CUtensorMap A, B;
  const uint64_t esz = 2;
  if (!tc::make_map(&A, a.w.slab, a.dt, a.V, a.R, a.Vp * esz, 64, 64)) return cudaErrorInvalidValue;
  if (!tc::make_map(&B, a.w.xc, a.dt, a.H, a.R, a.Hp * esz, 64, 64)) return cudaErrorInvalidValue;
  CUtensorMap C;  // dW for the TMA reduce-add (or store) of the epilogue
  const bool wide = a.R >= DW_WIDE_MIN_ROWS;
  if (a.dW_dt == FLCE_F32) {
    if (!tc::make_map(&C, a.dW, FLCE_F32, a.H, a.V, a.H * 4, wide ? 16 : 32, 32,
                      wide ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {  // same-dtype dW: 32-column boxes of 16-bit values, added (or stored) by the TMA unit
    if (!tc::make_map(&C, a.dW, a.dW_dt, a.H, a.V, a.H * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  const int64_t vt = (a.V + 255) / 256, ht = (a.H + 255) / 256;
  if (wide) return tc::launch_mode<tc::DW, 2>(a, chunk, s, A, B, C, vt * ((ht + 1) / 2));
  return tc::launch_mode<tc::DW, 1>(a, chunk, s, A, B, C, vt * ht);
}

bool bwd_merged_supported(const CallArgs& a) {
  return a.want_dX && a.want_dW && a.R >= DW_WIDE_MIN_ROWS && !(a.flags & FLCE_FLAG_SEPARATE_BWD);
}

namespace tc {
template <typename T>
cudaError_t launch_bwd_t(const CallArgs& a, int chunk, cudaStream_t s, const CUtensorMap (&m)[6],
                         int64_t items_max) {
  auto kern = k_gemm_bwd<T>;
  constexpr int smem = smem_bytes<DX, 2>();
  static std::atomic<int> max_pairs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs[dev].load(std::memory_order_relaxed) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (unsigned)(num_sms() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_pairs[dev].store(n, std::memory_order_relaxed);
  }
  const int mp = max_pairs[dev].load(std::memory_order_relaxed);
  const int64_t pairs = items_max < mp ? items_max : mp;
  if (pairs <= 0) return cudaSuccess;
  // the queue counter starts at zero for every launch
  e = cudaMemsetAsync(&a.w.ctrl->queue, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(2 * (unsigned)pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], m[5], a, chunk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace tc

cudaError_t launch_bwd_tc(const CallArgs& a, int chunk, cudaStream_t s) {
  CUtensorMap m[6];
  const uint64_t esz = 2;
  // dX: A = slab K-major, B = W MN-major, C = the two fp32 accumulator buffers [2R, H]
  if (!tc::make_map(&m[0], a.w.slab, a.dt, a.V, a.R, a.Vp * esz, 64, 128)) return cudaErrorInvalidValue;
  if (!tc::make_map(&m[1], a.W, a.dt, a.H, a.V, a.H * esz, 64, 64)) return cudaErrorInvalidValue;
  if (!tc::make_map(&m[2], a.w.dxacc, FLCE_F32, a.H, 2 * a.R, a.H * 4, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // dW: A = slab^T MN-major, B = Xc MN-major, C = dW (fp32 16-column or 16-bit 32-column boxes)
  if (!tc::make_map(&m[3], a.w.slab, a.dt, a.V, a.R, a.Vp * esz, 64, 64)) return cudaErrorInvalidValue;
  if (!tc::make_map(&m[4], a.w.xc, a.dt, a.H, a.R, a.Hp * esz, 64, 64)) return cudaErrorInvalidValue;
  if (a.dW_dt == FLCE_F32) {
    if (!tc::make_map(&m[5], a.dW, FLCE_F32, a.H, a.V, a.H * 4, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  } else {
    if (!tc::make_map(&m[5], a.dW, a.dW_dt, a.H, a.V, a.H * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  const int64_t ht2 = ((a.H + 255) / 256 + 1) / 2;
  const int64_t items = tc::DX_MAX_SPLITS * ((a.R + 255) / 256) * ht2 + ((a.V + 255) / 256) * ht2;
  if (a.dt == FLCE_BF16) return tc::launch_bwd_t<__nv_bfloat16>(a, chunk, s, m, items);
  return tc::launch_bwd_t<__half>(a, chunk, s, m, items);
}

}  // namespace flce
