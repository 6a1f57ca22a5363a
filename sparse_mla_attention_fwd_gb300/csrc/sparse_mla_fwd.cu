// Sparse MLA attention forward (DSA top-k) for sm_103a.
//
// Each query token t attends to its own list of top-k slots into one shared latent KV
// (h_kv = 1; K = kv[:, :d_qk], V = kv[:, :d_v]).  A slot j counts iff j < L_t and
// 0 <= idx[t][j] < s_kv, where L_t is the caller's topk_length[t] clamped to [0, topk], or topk
// when no topk_length is given.  Rows with no counted slot return O = 0, lse = +inf,
// max_logits = -inf (FlashMLA PR #196, "Correctness notes").  The optional per-head attention
// sink is a value-less virtual key in the softmax denominator (FlashMLA PR #198, "Summary"
// item 2).
//
// Work item = (token, group of 64 heads).  The kernel is persistent: one CTA per SM walks a
// static round-robin list of items, and every role streams through the same sequence of
// 64-key blocks, so one item's tail overlaps the next item's head.  A row's counted slots are
// packed into dense blocks, so it costs max(ceil(n_counted / 64), 1) blocks: trailing padding
// costs nothing (the fix of FlashMLA PR #196, "Fix") and neither do invalid entries inside the
// row.
//
// Warp roles (512 threads, 16 warps = 4 per SM sub-partition, warp w on sub-partition w % 4):
//   warps 0,1,3,8,9     gather    : TMA gather4 of the selected KV rows (whole rows: measured
//                                   ~45% faster per byte than half rows) into a 2-stage ring,
//                                   each stage handed over in four column groups.  A slot
//                                   without a counted index carries row coordinate -1, so TMA
//                                   zero-fills it and its index is never an address.
//   warps 4-7           softmax   : online exp2 softmax on S read as 16x256b TMEM fragments
//                                   (every lane holds 2 heads x 16 keys), P -> smem, lazy O
//                                   rescale, epilogue (sink, normalise, write O / lse / max).
//   warp 2              QK issuer : TMEM allocation, Q tile loads, S = QK^T.
//   warp 11             PV issuer : O^T += V^T P^T.
//   warp 10             scheduler : per row, one pass over its index list that packs the
//                                   counted slots into 64-slot blocks (resolved TMA row
//                                   coordinates + validity mask + first/last flags) in a shared
//                                   16-deep ring.  It runs ahead, so index loads never sit on
//                                   the critical path.
//   warps 12-15         V^T       : copy value columns 0..255 of each gathered block into TMEM
//                                   as V^T (ldmatrix.trans -> tcgen05.st) and issue gathers.
// setmaxnreg gives the softmax warpgroup 200 registers and the other three 104.
// Tensor-core work per 64-key block:
//   S[64 heads x 64 keys]  = Q_g . K_blk^T        (M=64, N=64, K=d_qk; both K-major SW128)
//   O^T[512 x 64 heads]   += V_blk^T . P^T        (4 x M=128, N=64, K=64; V^T of value columns
//                                                  256..511 read MN-major straight out of the
//                                                  gathered block, of columns 0..255 out of
//                                                  TMEM)
// TMEM: O^T in columns [0,256), S double buffer in [256,384), V^T double buffer (value columns
// 0..255) in [384,512).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kBlockN = 64;            // keys per k-block
constexpr int kGroupHeads = 64;        // heads per work item
constexpr int kDv = 512;               // value width (first d_v columns of each kv row)
// 16 warps = 4 per SM sub-partition (warp w runs on sub-partition w % 4).  S = QK^T and
// O^T += V^T P^T are issued by two different threads: the tensor unit interleaves two
// independent issue streams without the dead time a single issuer leaves between chains (it is
// blocked inside each chain's issue until the chain has nearly drained, then has to find the
// next ready chain).  The fourth warpgroup (warps 12-15, TMEM lane quadrants 0-3) copies V^T
// into TMEM and gathers; registers are rebalanced towards the softmax warpgroup.
constexpr int kThreads = 512;
constexpr int kVtWarp0 = 12;
constexpr int kSoftmaxRegs = 200;      // setmaxnreg split of the 512-thread kernel: 128 x 200
constexpr int kOtherRegs = 104;        // + 384 x 104 = 65536 = 512 threads x 128 at launch
constexpr int kGatherWarps = 5;        // warps 0, 1, 3, 8, 9
constexpr int kSoftmaxWarp0 = 4;       // warps 4-7 (TMEM lane quadrants 0-3)
constexpr int kQkWarp = 2;             // QK issuer; also allocates TMEM and loads Q tiles
constexpr int kPvWarp = 11;            // PV issuer
constexpr int kSchedWarp = 10;
constexpr int kRing = 16;              // scheduler ring depth (blocks)
constexpr int kRingConsumers = kGatherWarps + 4 + 2 + 4;   // gather, softmax, 2 issuers, V^T
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O^T: 4 chunks x 64 columns
constexpr uint32_t kTmemS = 256;       // S buffers: 256 + 64*b
constexpr uint32_t kTmemVT = 384;      // V^T of value chunks 0-1: 2 buffers x 2 chunks x 32 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;   // rescale O only when the running max grows by > 2^8
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // every device wait gives up after 2 s

// kEndOfWork marks the ring entry after the last block of the CTA's last work unit.
enum : uint32_t { kFirstBlock = 1u, kLastBlock = 2u, kEndOfWork = 4u };

__device__ int g_device_status = 0;    // SMLA_ERR_DEVICE_TIMEOUT once any wait gave up

// Scratch of the allocation-free split-KV entry point (sparse_mla_fwd_paged_splitkv_static):
// 32 MiB.  Each (row, head group, range) unit takes 131840 bytes of partial O and statistics,
// so up to 254 units fit, e.g. 8 rows x 2 head groups x 15 ranges.  Every unit writes its
// whole partial result before the merge reads it, so no part of it has to start at zero.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_splitkv_scratch[kStaticScratchBytes];

#ifdef SMLA_TRACE
// Pipeline trace (debug builds only): SM clock stamps of each block's events in CTA 0.
constexpr int kTraceBlocks = 256;
enum TraceEvent {
  kTrRing, kTrGatherIssue, kTrQkIssue, kTrSReady, kTrPReady, kTrPvIssue, kTrEpilogue,
  kTrSLoaded, kTrSent, kTrVtStart, kTrVtWait0, kTrVtEnd, kTrEvents
};
__device__ long long g_trace[kTraceBlocks][kTrEvents];
__device__ __forceinline__ void trace(int64_t b, int ev) {
  if (blockIdx.x == 0 && b < kTraceBlocks) g_trace[b][ev] = clock64();
}
#define SMLA_TRACE_EVENT(b, ev) trace((b), (ev))
#define SMLA_TRACE_EVENT_IF(cond, b, ev) \
  do {                                   \
    if (cond) trace((b), (ev));          \
  } while (0)
#else
#define SMLA_TRACE_EVENT(b, ev) ((void)0)
#define SMLA_TRACE_EVENT_IF(cond, b, ev) ((void)0)
#endif

struct FwdParams {
  const int32_t* indices;      // [s_q, topk]
  const int32_t* topk_length;  // [s_q] or null
  const float* attn_sink;      // [h_q] or null
  __nv_bfloat16* out;          // [s_q, h_q, d_v]
  float* lse;                  // [s_q, h_q]
  float* max_logits;           // [s_q, h_q]
  float sm_scale;
  int64_t s_q;
  int64_t s_kv;                // flat: rows of kv; paged: per-request length when seqlens_k null
  int h_q;
  int topk;
  int n_groups;                // h_q / 64
  int64_t n_items;             // s_q * n_groups
  // paged KV cache
  const int32_t* block_table;  // [n_req, max_blocks]
  const int32_t* seqlens_k;    // [n_req] or null
  int max_blocks;
  int page_block;
  int s_q_per_req;
  int64_t pool_rows;           // rows the KV tensor map covers
  // split-KV: each item's slot list is cut into n_split ranges, one work unit each, whose
  // partial results go to part_o [unit][64 heads][512] (unnormalised O) and part_stats
  // [unit][3][64] (exponent offset m in log2 units, sum l, max of sm_scale * q.k)
  int n_split;
  float* part_o;
  float* part_stats;
};

// One 64-key block as resolved by the scheduler warp.
struct BlockDesc {
  int32_t rows[kBlockN];       // TMA row coordinate per slot, -1 when the slot does not count
  uint32_t mask[2];            // validity bits of slots 0-31 / 32-63
  int32_t item;                // work item this block belongs to
  uint32_t flags;              // kFirstBlock | kLastBlock, or kEndOfWork alone
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  a = (a + 1023) & ~uintptr_t(1023);
  return reinterpret_cast<uint8_t*>(a);
}

// Wait that records a device timeout and lets the caller carry on (never hangs, never traps).
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint64_t limit_ns) {
  if (!mbar_wait_bounded(bar, parity, abort, limit_ns)) {
    *abort = 1;
    atomicExch(&g_device_status, static_cast<int>(SMLA_ERR_DEVICE_TIMEOUT));
  }
}

// Bounded wait that ignores the abort flag: used only to let this CTA's own asynchronous
// copies / MMAs finish before it releases TMEM or exits.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  int never = 0;
  if (!mbar_wait_bounded(bar, parity, &never, limit_ns))
    atomicExch(&g_device_status, static_cast<int>(SMLA_ERR_DEVICE_TIMEOUT));
}

template <bool PAGED>
__device__ __forceinline__ int64_t row_kv_len(const FwdParams& p, int64_t t) {
  if (!PAGED) return p.s_kv;
  const int64_t req = t / p.s_q_per_req;
  return p.seqlens_k ? static_cast<int64_t>(__ldg(p.seqlens_k + req)) : p.s_kv;
}

// Validity predicate of one slot value (FlashMLA PR #196, "Fix": 0 <= idx < s_kv).  For a
// paged cache the position must also map to an entry of the request's block table.
template <bool PAGED>
__device__ __forceinline__ bool slot_ok(const FwdParams& p, int v, int64_t kv_len) {
  if (v < 0 || static_cast<int64_t>(v) >= kv_len) return false;
  if (PAGED && v / p.page_block >= p.max_blocks) return false;
  return true;
}

// TMA row coordinate of a valid slot value.
template <bool PAGED>
__device__ __forceinline__ int kv_row_of(const FwdParams& p, int64_t t, int v) {
  if (!PAGED) return v;
  const int64_t req = t / p.s_q_per_req;
  const int64_t page = __ldg(p.block_table + req * p.max_blocks + v / p.page_block);
  const int64_t row = page * p.page_block + v % p.page_block;
  return (page < 0 || row >= p.pool_rows) ? -1 : static_cast<int>(row);
}

// SPLIT: work units are (item, slot range); the epilogue writes the unit's partial result to
// the split-KV workspace instead of O / lse / max_logits (a second kernel merges the ranges).
template <int D_QK, bool DYNAMIC, bool PAGED, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_fwd_kernel(const __grid_constant__ CUtensorMap q_map,
                          const __grid_constant__ CUtensorMap kv_map, const FwdParams p) {
  constexpr int kChunks = D_QK / 64;                 // 128-byte column chunks of a row
  constexpr uint32_t kTileBytes = kChunks * 8192u;   // 64 rows x D_QK bf16 (= Q tile = stage)
  constexpr int kQkSteps = D_QK / 16;
  // P^T (64 heads x 64 keys bf16, 8 KB) of block b lives in the rope chunk (columns 512..575)
  // of stage b%2 when there is one -- that chunk is dead once S = QK^T has been computed --
  // and in a separate double buffer otherwise.
  constexpr bool kPInStage = (kChunks > 8);
  // A stage is handed over in kGroups groups of columns: group g holds column chunks 2g and
  // 2g+1 (the last group also the rope chunk).  PV's M-chunk g reads exactly group g's value
  // columns, so group g of a stage is refilled as soon as PV M-chunk g of the block before has
  // completed, and S = QK^T of the new block starts on group 0 while later groups are in flight.
  constexpr int kGroups = 4;
  // PV reads value chunks 0-1 (columns 0..255) as V^T out of TMEM, double-buffered in the 128
  // columns that O^T and S leave free; chunks 2-3 it reads from the stage as usual.  The V^T
  // warps copy column groups 0-1 of a stage into TMEM (ldmatrix.trans -> tcgen05.st) as soon
  // as they land, so those groups are released once S = QK^T and the copy have read them, well
  // before PV; the gather of groups 0-1 of block b+2 then overlaps PV of block b, and QK(b+2)
  // streams through them while groups 2-3 are in flight.  With a rope chunk, P^T lives in it,
  // so group 3 goes back only after PV's last M-chunk.

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kTileBytes;                  // stage s at sKV + s * kTileBytes
  uint8_t* sPbuf = smem + 3 * kTileBytes;            // used when !kPInStage: 2 x 8 KB

  __shared__ __align__(16) BlockDesc ring[kRing];
  __shared__ __align__(8) uint64_t bar_ring_full[kRing], bar_ring_empty[kRing];
  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty;
  __shared__ __align__(8) uint64_t bar_kv_full[2][kGroups], bar_kv_empty[2][kGroups];
  __shared__ __align__(8) uint64_t bar_s_full[2], bar_p_full[2], bar_o_done[2], bar_o_free;
  __shared__ __align__(8) uint64_t bar_final_qk, bar_final_pv;
  __shared__ __align__(8) uint64_t bar_vt_full[2][2], bar_vt_free[2][2];   // [buffer][chunk]
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float s_alpha[kGroupHeads];
  __shared__ float s_inv[kGroupHeads];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort = &abort_flag;
  constexpr uint64_t lim = kDefaultWaitLimitNs;
  // Work units: an item (token, 64-head group) or, with SPLIT, an (item, slot range) pair.  One
  // CTA per SM walks the units blockIdx.x, blockIdx.x + gridDim.x, ...  The scheduler warp
  // publishes their blocks in that order, followed by an end-of-work entry; every role but the
  // QK issuer simply follows the block ring until that entry.
  const int64_t n_units = SPLIT ? p.n_items * p.n_split : p.n_items;
  const int64_t n_my_items = n_units > blockIdx.x ? (n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto item_of_unit = [&](int64_t u) -> int64_t { return SPLIT ? u / p.n_split : u; };

  auto p_addr = [&](int b) -> uint8_t* {
    if constexpr (kPInStage) return sKV + (b & 1) * kTileBytes + 8 * 8192;
    else return sPbuf + (b & 1) * 8192;
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int r = 0; r < kRing; ++r) {
      mbar_init(smem_u32(&bar_ring_full[r]), 1);
      mbar_init(smem_u32(&bar_ring_empty[r]), kRingConsumers);
    }
    mbar_init(smem_u32(&bar_q_full), 1);
    mbar_init(smem_u32(&bar_q_empty), 1);
    for (int s = 0; s < 2; ++s) {
      for (int g = 0; g < kGroups; ++g) {
        mbar_init(smem_u32(&bar_kv_full[s][g]), 1);
        // groups 0-1 are released by S = QK^T (one commit) and the four V^T warps, groups 2-3
        // by PV (one commit)
        mbar_init(smem_u32(&bar_kv_empty[s][g]), g < 2 ? 5 : 1);
      }
      mbar_init(smem_u32(&bar_s_full[s]), 1);
      mbar_init(smem_u32(&bar_p_full[s]), 128);
      mbar_init(smem_u32(&bar_o_done[s]), 1);
    }
    mbar_init(smem_u32(&bar_o_free), 128);
    mbar_init(smem_u32(&bar_final_qk), 1);
    mbar_init(smem_u32(&bar_final_pv), 1);
    for (int v = 0; v < 4; ++v) {
      mbar_init(smem_u32(&bar_vt_full[v >> 1][v & 1]), 4);
      mbar_init(smem_u32(&bar_vt_free[v >> 1][v & 1]), 1);
    }
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Roles.  The softmax warpgroup comes first so that, in the 512-thread kernel, its code is
  // dominated by the register increase and every other role by the decrease.
  if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4) {
    reg_alloc<kSoftmaxRegs>();
    // ======================================================== softmax / correction / epilogue
    const int q = warp - kSoftmaxWarp0;          // TMEM lane quadrant 0..3
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // 16x256b fragments of S (M=64 layout: heads 16q..16q+15 in lanes 0-15 of quadrant q):
    // this thread holds heads hA = 16q + lane/4 and hB = hA + 8, columns 8i + 2(lane&3) + {0,1}.
    const int hA = 16 * q + (lane >> 2);
    const int hB = hA + 8;
    const int cpair = 2 * (lane & 3);
    const bool quad_leader = (lane & 3) == 0;
    const float c = p.sm_scale * kLog2e;
    float m_used[2] = {-INFINITY, -INFINITY};    // running exponent offsets (log2 units)
    float s_max[2] = {-INFINITY, -INFINITY};     // running max of raw q.k
    float l_sum[2] = {0.f, 0.f};
    for (int64_t b = 0; !*abort; ++b) {
      {
        const int r = static_cast<int>(b % kRing);
        const int sb = static_cast<int>(b & 1);
        wait_or_flag(smem_u32(&bar_ring_full[r]), (b / kRing) & 1, abort, lim);
        const uint32_t mask_lo = ring[r].mask[0], mask_hi = ring[r].mask[1];
        const uint32_t flags = ring[r].flags;
        const int64_t item = ring[r].item;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_ring_empty[r]));
        if (flags & kEndOfWork) break;
        const bool more = (flags & kLastBlock) == 0;
        const bool first = (flags & kFirstBlock) != 0;
        if (first) {
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            m_used[x] = -INFINITY;
            s_max[x] = -INFINITY;
            l_sum[x] = 0.f;
          }
        }

        wait_or_flag(smem_u32(&bar_s_full[sb]), (b >> 1) & 1, abort, lim);
        tc_fence_after();
        SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, b, kTrSReady);
        float sv[32];   // sv[4i+0/1] = head hA, cols 8i+cpair+0/1; sv[4i+2/3] = head hB
#pragma unroll
        for (int i8 = 0; i8 < 8; ++i8) {
          uint32_t r4[4];
          tmem_ld_16x256b(tmem + lane_base + kTmemS + 64 * sb + 8 * i8, r4);
#pragma unroll
          for (int e = 0; e < 4; ++e) sv[4 * i8 + e] = __uint_as_float(r4[e]);
        }
        tmem_ld_wait();

        if ((mask_lo & mask_hi) != 0xffffffffu) {
          // this thread's columns are 8i + cpair + {0,1}: shift its bits down once
          const uint32_t mlo = mask_lo >> cpair, mhi = mask_hi >> cpair;
#pragma unroll
          for (int i8 = 0; i8 < 8; ++i8) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const bool ok = (((i8 < 4 ? mlo : mhi) >> (8 * (i8 & 3) + e)) & 1u) != 0u;
              sv[4 * i8 + e] = ok ? sv[4 * i8 + e] : -INFINITY;
              sv[4 * i8 + 2 + e] = ok ? sv[4 * i8 + 2 + e] : -INFINITY;
            }
          }
        }
        float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int i8 = 0; i8 < 8; ++i8) {
          bm[0] = fmaxf(bm[0], fmaxf(sv[4 * i8], sv[4 * i8 + 1]));
          bm[1] = fmaxf(bm[1], fmaxf(sv[4 * i8 + 2], sv[4 * i8 + 3]));
        }
        float alpha[2] = {1.f, 1.f};
        bool need_rescale = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          bm[x] = fmaxf(bm[x], __shfl_xor_sync(0xffffffffu, bm[x], 1));
          bm[x] = fmaxf(bm[x], __shfl_xor_sync(0xffffffffu, bm[x], 2));
          s_max[x] = fmaxf(s_max[x], bm[x]);
          const float bm2 = bm[x] * c;
          if (bm2 > m_used[x] + kRescaleLog2) {
            alpha[x] = fast_exp2(m_used[x] - bm2);   // 0 when m_used was -inf
            m_used[x] = bm2;
            need_rescale = true;
          }
        }
        // P as bf16 into the P^T operand tile ([64 heads][64 keys], 128-byte swizzle).  Its
        // previous user (block b-2) finished its PV before the stage was refilled for block b,
        // which S(b) being ready already implies when P^T lives in the stage's rope chunk.  The
        // separate P^T buffer (no rope chunk) has no such link -- PV's last M-chunks read TMEM,
        // not the stage -- so PV(b-2) is waited for here.  Masked slots hold
        // -inf and give exp2(-inf) = 0; a row whose offset is still -inf has no valid slot yet,
        // and any finite offset then yields 0 as well.
        if (!kPInStage && b >= 2) wait_or_flag(smem_u32(&bar_o_done[sb]), ((b - 2) >> 1) & 1, abort, lim);
        const float neg_m0 = m_used[0] == -INFINITY ? 0.f : -m_used[0];
        const float neg_m1 = m_used[1] == -INFINITY ? 0.f : -m_used[1];
        uint8_t* ptile = p_addr(static_cast<int>(b));
        const int swA = hA & 7, swB = hB & 7;
        float ls[2] = {0.f, 0.f};
        uint8_t* prowA = ptile + hA * 128 + 2 * cpair;
        uint8_t* prowB = ptile + hB * 128 + 2 * cpair;
#pragma unroll
        for (int i8 = 0; i8 < 8; ++i8) {
          const float p0 = fast_exp2(fmaf(sv[4 * i8], c, neg_m0));
          const float p1 = fast_exp2(fmaf(sv[4 * i8 + 1], c, neg_m0));
          const float p2 = fast_exp2(fmaf(sv[4 * i8 + 2], c, neg_m1));
          const float p3 = fast_exp2(fmaf(sv[4 * i8 + 3], c, neg_m1));
          ls[0] += p0 + p1;
          ls[1] += p2 + p3;
          *reinterpret_cast<uint32_t*>(prowA + ((i8 ^ swA) << 4)) = pack_bf16x2(p0, p1);
          *reinterpret_cast<uint32_t*>(prowB + ((i8 ^ swB) << 4)) = pack_bf16x2(p2, p3);
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          ls[x] += __shfl_xor_sync(0xffffffffu, ls[x], 1);
          ls[x] += __shfl_xor_sync(0xffffffffu, ls[x], 2);
          l_sum[x] = fmaf(l_sum[x], alpha[x], ls[x]);
        }
        // O^T holds earlier blocks of this item only when this is not the item's first block;
        // it must then be rescaled before PV of this block if some head's offset moved.
        const bool any_rescale = named_bar_or(1, 128, need_rescale && !first);
        if (any_rescale) {
          // PV of the previous block must be complete before O^T is touched
          wait_or_flag(smem_u32(&bar_o_done[(b - 1) & 1]), ((b - 1) >> 1) & 1, abort, lim);
          if (quad_leader) {
            s_alpha[hA] = alpha[0];
            s_alpha[hB] = alpha[1];
          }
          named_bar_sync(2, 128);
          tc_fence_after();
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              uint32_t rg[16];
              const uint32_t addr = tmem + lane_base + kTmemO + 64 * m + 16 * i4;
              tmem_ld16(addr, rg);
              tmem_ld_wait();
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                rg[jj] = __float_as_uint(__uint_as_float(rg[jj]) * s_alpha[16 * i4 + jj]);
              tmem_st16(addr, rg);
            }
          }
          tmem_st_wait();
          named_bar_sync(2, 128);                  // s_alpha is reused by the next rescale
        }
        fence_proxy_async_smem();
        tc_fence_before();
        SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, b, kTrPReady);
        mbar_arrive(smem_u32(&bar_p_full[sb]));

        if (!more) {
          // ---- epilogue of this item (or, with SPLIT, of this unit)
          const int64_t unit = item;
          const int64_t it_ = item_of_unit(unit);
          const int64_t t = it_ / p.n_groups;
          const int g = static_cast<int>(it_ % p.n_groups);
          if constexpr (SPLIT) {
            // partial result: exponent offset, sum and max per head; unnormalised O^T below
            if (quad_leader) {
              float* st = p.part_stats + unit * (3 * kGroupHeads);
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                const int h = x ? hB : hA;
                const bool empty = !(l_sum[x] > 0.f);
                st[h] = empty ? -INFINITY : m_used[x];
                st[kGroupHeads + h] = empty ? 0.f : l_sum[x];
                st[2 * kGroupHeads + h] = empty ? -INFINITY : s_max[x] * p.sm_scale;
              }
            }
          } else if (quad_leader) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const int h = x ? hB : hA;
              const int head = g * kGroupHeads + h;
              const bool empty = !(l_sum[x] > 0.f);
              float den = l_sum[x];
              if (p.attn_sink) den += exp2f(fmaf(__ldg(p.attn_sink + head), kLog2e, -m_used[x]));
              s_inv[h] = empty ? 0.f : 1.f / den;
              const int64_t o = t * p.h_q + head;
              p.lse[o] = empty ? INFINITY : (m_used[x] + log2f(l_sum[x])) * kLn2;
              p.max_logits[o] = empty ? -INFINITY : s_max[x] * p.sm_scale;
            }
          }
          wait_or_flag(smem_u32(&bar_o_done[sb]), (b >> 1) & 1, abort, lim);
          named_bar_sync(2, 128);
          tc_fence_after();
          SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, b, kTrEpilogue);
          // O goes out with direct stores: the 32 lanes of a warp hold 32 consecutive d of one
          // head (64 contiguous bytes of bf16, or 128 of fp32 partials).  (Staging through
          // shared memory for TMA tensor stores measured slower: the stores queue behind the
          // gathers in the TMA unit.)
          __nv_bfloat16* out_t = p.out + (t * p.h_q + g * kGroupHeads) * static_cast<int64_t>(kDv);
          float* part_t = SPLIT ? p.part_o + unit * (kGroupHeads * kDv) : nullptr;
#pragma unroll 1
          for (int m = 0; m < 4; ++m) {
            const int dcol = 128 * m + 32 * q + lane;   // column d of this lane
#pragma unroll 1
            for (int i4 = 0; i4 < 4; ++i4) {
              uint32_t rg[16];
              tmem_ld16(tmem + lane_base + kTmemO + 64 * m + 16 * i4, rg);
              tmem_ld_wait();
              if (m == 3 && i4 == 3) {
                // all of O^T has been read: the next item's first PV may overwrite it
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_o_free));
              }
              if constexpr (SPLIT) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) part_t[(16 * i4 + jj) * kDv + dcol] = __uint_as_float(rg[jj]);
              } else {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                  const float inv = s_inv[16 * i4 + jj];
                  const float val = (inv == 0.f) ? 0.f : __uint_as_float(rg[jj]) * inv;
                  out_t[(16 * i4 + jj) * kDv + dcol] = __float2bfloat16_rn(val);
                }
              }
            }
          }
        }
      }
    }
  } else {
    reg_dealloc<kOtherRegs>();
    if (warp == kSchedWarp) {
      // ======================================================== scheduler
      // Per row, a parallel scan first finds the last counted slot (j < L_t, 0 <= idx < s_kv) and
      // the number of counted slots.  A row whose counted slots form a dense prefix (the usual
      // case: front-packed lists, -1 or INT_MAX padding) is cut into blocks straight from its
      // slot list, so trailing padding costs nothing (FlashMLA PR #196, "Fix").  Any other row is
      // packed: its counted slots go, in slot order, into dense blocks, so invalid entries inside
      // the row cost nothing either.  The result does not depend on the packing (it is invariant
      // under permuting slots and inserting invalid ones; the oracle's pins check both).  A row
      // costs max(ceil(n_counted / 64), 1) blocks, and every role walks the same block stream.
      const uint32_t lanes_below = (1u << lane) - 1u;
      auto acquire = [&](int64_t blk) {
        if (blk >= kRing)
          wait_or_flag(smem_u32(&bar_ring_empty[blk % kRing]), ((blk / kRing) - 1) & 1, abort, lim);
      };
      auto publish = [&](int64_t blk, uint32_t m0, uint32_t m1, uint32_t flags, int64_t item) {
        const int r = static_cast<int>(blk % kRing);
        if (lane == 0) {
          ring[r].mask[0] = m0;
          ring[r].mask[1] = m1;
          ring[r].item = static_cast<int32_t>(item);
          ring[r].flags = flags;
        }
        __syncwarp();
        if (lane == 0) {
          SMLA_TRACE_EVENT(blk, kTrRing);
          mbar_arrive(smem_u32(&bar_ring_full[r]));
        }
      };
      int64_t b = 0;
      for (int64_t unit = blockIdx.x; unit < n_units && !*abort; unit += gridDim.x) {
        const int64_t item = unit;   // what the ring carries: the unit (the item itself unless SPLIT)
        const int64_t t = item_of_unit(unit) / p.n_groups;
        const int32_t* idx_row = p.indices + t * static_cast<int64_t>(p.topk);
        const int64_t kv_len = row_kv_len<PAGED>(p, t);
        int Lr = DYNAMIC ? min(max(__ldg(p.topk_length + t), 0), p.topk) : p.topk;
        if constexpr (SPLIT) {
          // this unit's share of the row: range `split` of n_split 64-aligned ranges of [0, L_t)
          const int split = static_cast<int>(unit % p.n_split);
          const int span = ((Lr + p.n_split - 1) / p.n_split + kBlockN - 1) / kBlockN * kBlockN;
          const int j0 = min(split * span, Lr);
          idx_row += j0;
          Lr = min(Lr - j0, span);
        }
        int last = -1, cnt = 0;
        if constexpr (PAGED) {
          // Decode-shaped work has few blocks per CTA, so the scan's load latency is exposed:
          // keep eight 32-slot chunks of loads in flight.  (On the prefill paths, which are
          // throughput-bound, this form measured slower.)
          for (int j0 = 0; j0 < Lr; j0 += 8 * 32) {
            int vals[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = j0 + 32 * u + lane;
              vals[u] = j < Lr ? __ldg(idx_row + j) : -1;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = j0 + 32 * u + lane;
              if (j < Lr && slot_ok<PAGED>(p, vals[u], kv_len)) {
                last = j;
                ++cnt;
              }
            }
          }
        } else {
          for (int j = lane; j < Lr; j += 32)
            if (slot_ok<PAGED>(p, __ldg(idx_row + j), kv_len)) {
              last = j;
              ++cnt;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
          cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        }
        const int L = last + 1;
        if (cnt == L) {
          // dense prefix: block k holds slots 64k .. 64k+63 of the list
          const int nblk = max((L + kBlockN - 1) / kBlockN, 1);
          for (int k = 0; k < nblk && !*abort; ++k, ++b) {
            const int r = static_cast<int>(b % kRing);
            acquire(b);
            uint32_t m[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int slot = k * kBlockN + 32 * h + lane;
              int coord = -1;
              if (slot < L) {
                const int v = __ldg(idx_row + slot);
                if (slot_ok<PAGED>(p, v, kv_len)) coord = kv_row_of<PAGED>(p, t, v);
              }
              ring[r].rows[32 * h + lane] = coord;
              m[h] = __ballot_sync(0xffffffffu, coord >= 0);
            }
            publish(b, m[0], m[1], (k == 0 ? kFirstBlock : 0u) | (k == nblk - 1 ? kLastBlock : 0u), item);
          }
        } else {
          // packing pass over [0, L): the indices were just read and come from L1
          const int64_t b0 = b;
          int count = 0;               // counted slots packed so far
          int64_t acquired = b0 - 1;   // last block whose ring slot is held
          int64_t published = b0;      // next block to publish
          for (int j0 = 0; j0 < L && !*abort; j0 += 32) {
            const int slot = j0 + lane;
            int coord = -1;
            if (slot < L) {
              const int v = __ldg(idx_row + slot);
              if (slot_ok<PAGED>(p, v, kv_len)) coord = kv_row_of<PAGED>(p, t, v);
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, coord >= 0);
            if (bal == 0u) continue;
            const int n = __popc(bal);
            const int64_t newest = b0 + (count + n - 1) / kBlockN;   // block of the newest slot
            while (acquired < newest) acquire(++acquired);
            if (coord >= 0) {
              const int pos = count + __popc(bal & lanes_below);
              ring[(b0 + pos / kBlockN) % kRing].rows[pos % kBlockN] = coord;
            }
            count += n;
            __syncwarp();
            // every block before the newest one is full and has a successor
            for (; published < newest; ++published)
              publish(published, 0xffffffffu, 0xffffffffu, published == b0 ? kFirstBlock : 0u, item);
          }
          // the block that holds the row's last counted slot (or one empty block) closes the item
          if (count == 0) acquire(++acquired);
          const int64_t lastb = b0 + (count > 0 ? (count - 1) / kBlockN : 0);
          const int fill = count - static_cast<int>(lastb - b0) * kBlockN;   // 0..64 slots used
          const int rl = static_cast<int>(lastb % kRing);
          for (int e = fill + lane; e < kBlockN; e += 32) ring[rl].rows[e] = -1;
          const uint32_t m0 = fill >= 32 ? 0xffffffffu : ((1u << fill) - 1u);
          const uint32_t m1 = fill >= 64 ? 0xffffffffu : (fill > 32 ? ((1u << (fill - 32)) - 1u) : 0u);
          __syncwarp();
          publish(lastb, m0, m1, (lastb == b0 ? kFirstBlock : 0u) | kLastBlock, item);
          b = lastb + 1;
        }
      }
      // every role stops at this entry
      acquire(b);
      publish(b, 0u, 0u, kEndOfWork, -1);
    } else if (warp < 2 || warp == 3 || warp == 8 || warp == 9 || warp >= kVtWarp0) {
      // ======================================================== gather (+ V^T copies)
      // TMA issue throughput grows with the number of issuing warps, so the 16 x (chunks of a
      // group) gather4 items of each column group are dealt round-robin over the gather warps:
      // warps 0, 1, 3, 8, 9 and the four V^T warps 12-15.
      constexpr int kGW = kGatherWarps + 4;
      // gather warp index 0..kGW-1: warps 0, 1, 3, 8, 9 -> 0..4, warps 12-15 -> 5..8
      const int gw = warp < 2 ? warp
                   : warp == 3 ? 2
                   : warp < kVtWarp0 ? warp - 5
                                     : warp - kVtWarp0 + kGatherWarps;
      const int it = gw + kGW * lane;                 // item within a group: (4-row group, chunk)
      const int grp = it & 15;
      const bool leader = (gw == 0 && lane == 0);
      // V^T copies (warps 12-15 only).  Warp 12+q fills TMEM lanes 32q..32q+31 of V^T chunks
      // 0-1 (value columns 128m..128m+127 = column group m of the stage) in buffer j&1.  For
      // each 16-row half hh and 16-key step x, ldmatrix.trans loads matrix i = keys 16x + 8(i>>1)
      // + 0..7 by columns 128m + 32q + 16hh + 8(i&1) + 0..7 (eight rows of distinct swizzle
      // phase: no bank conflicts); thread t then holds keys 16x + 8(i>>1) + 2(t&3) + {0,1} of
      // column (t>>2) (+8 for odd i), which is exactly what a 16x128b store puts at K positions
      // 2c, 2c+1 of TMEM column c = 8x + 4(i>>1) + (t&3): natural key order.  The copy of block
      // j comes in the middle of this warp's gathers for block j+1 and before those for block
      // j+2, which wait for it (through kv_empty).
      const bool vt_warp = warp >= kVtWarp0;
      auto copy_vt = [&](int64_t j) {
        const int q = warp - kVtWarp0;
        const int mat = lane >> 3, rr = lane & 7;
        const int s = static_cast<int>(j & 1);
        const uint32_t stage = smem_u32(sKV + s * kTileBytes) + (q >> 1) * 8192 +
                               static_cast<uint32_t>((8 * (mat >> 1) + rr) * 128);
        SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, j, kTrVtStart);
#pragma unroll 1
        for (int m = 0; m < 2; ++m) {
          // block j's group m has landed; PV of block j-2 has read V^T buffer j&1, chunk m
          wait_or_flag(smem_u32(&bar_kv_full[s][m]), (j >> 1) & 1, abort, lim);
          if (j >= 2) wait_or_flag(smem_u32(&bar_vt_free[s][m]), ((j - 2) >> 1) & 1, abort, lim);
          SMLA_TRACE_EVENT_IF(m == 0 && q == 0 && lane == 0, j, kTrVtWait0);
          tc_fence_after();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int u = 4 * (q & 1) + 2 * hh + (mat & 1);
            const uint32_t a0 = stage + 2 * m * 8192 + ((u ^ rr) << 4);
            uint32_t rg[16];
#pragma unroll
            for (int x = 0; x < 4; ++x)
              ldsm_x4_trans(a0 + 2048 * x, rg[4 * x], rg[4 * x + 1], rg[4 * x + 2], rg[4 * x + 3]);
            const uint32_t lanes = static_cast<uint32_t>(32 * q + 16 * hh) << 16;
            tmem_st_16x128b_x8(tmem + lanes + kTmemVT + 64 * s + 32 * m, rg);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bar_vt_full[s][m]));
            mbar_arrive(smem_u32(&bar_kv_empty[s][m]));
          }
        }
        SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, j, kTrVtEnd);
      };
      int64_t b = 0;
      for (; !*abort; ++b) {
        {
          const int r = static_cast<int>(b % kRing);
          const int s = static_cast<int>(b & 1);
          wait_or_flag(smem_u32(&bar_ring_full[r]), (b / kRing) & 1, abort, lim);
          const uint32_t fl = ring[r].flags;
          const int4 rr = *reinterpret_cast<const int4*>(&ring[r].rows[4 * grp]);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_ring_empty[r]));
          if (fl & kEndOfWork) break;
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const int c0 = 2 * g;
            const int nch = (g == kGroups - 1) ? kChunks - c0 : 2;
            // a V^T warp copies block b-1 between its gathers of groups 0-1 and 2-3 of block b:
            // groups 2-3 wait for PV(b-2), which the copy does not need
            if (vt_warp && g == 2 && b >= 1) copy_vt(b - 1);
            if (b >= 2) wait_or_flag(smem_u32(&bar_kv_empty[s][g]), ((b >> 1) - 1) & 1, abort, lim);
            if (leader) {
              if (g == 0) SMLA_TRACE_EVENT(b, kTrGatherIssue);
              mbar_arrive_expect_tx(smem_u32(&bar_kv_full[s][g]), nch * 8192u);
            }
            if (it < 16 * nch) {
              const int chunk = c0 + (it >> 4);
              tma_gather4(smem_u32(sKV + s * kTileBytes + chunk * 8192 + grp * 512), &kv_map, 64 * chunk,
                          rr.x, rr.y, rr.z, rr.w, smem_u32(&bar_kv_full[s][g]));
            }
          }
        }
      }
      // the V^T copy of the last block
      if (vt_warp && b >= 1 && !*abort) copy_vt(b - 1);
      // drain: the last fills of both stages have landed before this CTA may exit
      if (leader) {
        for (int64_t bb = (b >= 2 ? b - 2 : 0); bb < b; ++bb)
          for (int g = 0; g < kGroups; ++g)
            wait_drain(smem_u32(&bar_kv_full[bb & 1][g]), (bb >> 1) & 1, lim);
      }
    } else if (warp == kQkWarp) {
      // ======================================================== QK issuer (and Q tile loads)
      if (lane == 0) {
        constexpr uint32_t idesc_qk = make_idesc_bf16(64, kBlockN, false, false);
        const uint64_t qd0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint32_t kv_base = smem_u32(sKV);
        auto load_q = [&](int64_t i) {
          const int64_t item = item_of_unit(blockIdx.x + i * gridDim.x);
          const int64_t t = item / p.n_groups;
          const int g = static_cast<int>(item % p.n_groups);
          mbar_arrive_expect_tx(smem_u32(&bar_q_full), kTileBytes);
          const int qrow = static_cast<int>(t * p.h_q + g * kGroupHeads);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(smem_u32(sQ + c * 8192), &q_map, 64 * c, qrow, smem_u32(&bar_q_full));
        };
        int64_t q_loaded = 0;                      // Q tiles requested so far
        if (n_my_items > 0) {
          load_q(0);
          q_loaded = 1;
        }
        int64_t b = 0;
        for (int64_t i = 0; i < n_my_items && !*abort; ++i) {
          wait_or_flag(smem_u32(&bar_q_full), i & 1, abort, lim);
          for (bool more = true; more && !*abort; ++b) {
            const int r = static_cast<int>(b % kRing);
            const int s = static_cast<int>(b & 1);
            wait_or_flag(smem_u32(&bar_ring_full[r]), (b / kRing) & 1, abort, lim);
            more = (ring[r].flags & kLastBlock) == 0;
            mbar_arrive(smem_u32(&bar_ring_empty[r]));
            // S buffer s was last read by the softmax of block b-2
            if (b >= 2) wait_or_flag(smem_u32(&bar_p_full[s]), ((b - 2) >> 1) & 1, abort, lim);
            const uint64_t kd0 = make_sdesc_sw128(kv_base + s * kTileBytes, 16, 1024);
            // S = QK^T group by group, as the column groups of the stage land.  Groups 0 and 1
            // are waited for together: starting on group 0 while group 1 is still landing measured
            // ~1 % slower (more of the operand reads then overlap the fill of the same stage).
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              if (g == 0) {
                wait_or_flag(smem_u32(&bar_kv_full[s][0]), (b >> 1) & 1, abort, lim);
                wait_or_flag(smem_u32(&bar_kv_full[s][1]), (b >> 1) & 1, abort, lim);
              } else if (g > 1) {
                wait_or_flag(smem_u32(&bar_kv_full[s][g]), (b >> 1) & 1, abort, lim);
              }
              tc_fence_after();
              if (g == 0) SMLA_TRACE_EVENT(b, kTrQkIssue);
              const int ks_end = (g == kGroups - 1) ? kQkSteps : 8 * (g + 1);
#pragma unroll
              for (int ks = 8 * g; ks < ks_end; ++ks) {
                const uint32_t off16 = ((ks >> 2) * 8192 + (ks & 3) * 32) >> 4;
                umma_ss(tmem + kTmemS + 64 * s, qd0 + off16, kd0 + off16, idesc_qk, ks > 0 ? 1u : 0u);
              }
              // with V^T in TMEM, PV does not read groups 0-1 of the stage: S = QK^T releases them
              if (g < 2) umma_commit(smem_u32(&bar_kv_empty[s][g]));
            }
            umma_commit(smem_u32(&bar_s_full[s]));
            SMLA_TRACE_EVENT(b, kTrSLoaded);
          }
          // the next item's Q tile replaces this one once this item's last S = QK^T is done
          if (i + 1 < n_my_items && !*abort) {
            umma_commit(smem_u32(&bar_q_empty));
            wait_or_flag(smem_u32(&bar_q_empty), i & 1, abort, lim);
            load_q(i + 1);
            ++q_loaded;
          }
        }
        // drain: every MMA issued above completes before TMEM is released, and the last Q tile
        // requested has landed before the CTA may exit
        umma_commit(smem_u32(&bar_final_qk));
        wait_drain(smem_u32(&bar_final_qk), 0, lim);
        if (q_loaded > 0) wait_drain(smem_u32(&bar_q_full), (q_loaded - 1) & 1, lim);
      }
      __syncwarp();
    } else if (warp == kPvWarp) {
      // ======================================================== PV issuer
      if (lane == 0) {
        constexpr uint32_t idesc_pv = make_idesc_bf16(128, kGroupHeads, true, false);
        constexpr uint32_t idesc_pv_ts = make_idesc_bf16(128, kGroupHeads, false, false);
        const uint32_t kv_base = smem_u32(sKV);
        uint32_t units_started = 0;
        for (int64_t b = 0; !*abort; ++b) {
          {
            const int r = static_cast<int>(b % kRing);
            const int sb = static_cast<int>(b & 1);
            wait_or_flag(smem_u32(&bar_ring_full[r]), (b / kRing) & 1, abort, lim);
            const uint32_t fl = ring[r].flags;
            mbar_arrive(smem_u32(&bar_ring_empty[r]));
            if (fl & kEndOfWork) break;
            const bool first = (fl & kFirstBlock) != 0;
            wait_or_flag(smem_u32(&bar_p_full[sb]), (b >> 1) & 1, abort, lim);
            // the epilogue of the previous unit has read all of O^T
            if (first) {
              if (units_started > 0) wait_or_flag(smem_u32(&bar_o_free), (units_started - 1) & 1, abort, lim);
              ++units_started;
            }
            tc_fence_after();
            SMLA_TRACE_EVENT(b, kTrPvIssue);
            // descriptor start addresses advance in 16-byte units (low 14 bits)
            const uint64_t b0 = make_sdesc_sw128(smem_u32(p_addr(static_cast<int>(b))), 16, 1024);
            // M-chunks 2-3 from the stage first (that frees its column groups 2-3), then 0-1 from
            // V^T buffer b&1 in TMEM
            const uint64_t a0 = make_sdesc_sw128(kv_base + sb * kTileBytes, 8192, 1024);
#pragma unroll
            for (int m = 2; m < 4; ++m) {
#pragma unroll
              for (int ks = 0; ks < kBlockN / 16; ++ks)
                umma_ss(tmem + kTmemO + 64 * m, a0 + ((2 * m * 8192 + ks * 2048) >> 4),
                        b0 + ((ks * 32) >> 4), idesc_pv, (!first || ks > 0) ? 1u : 0u);
              // with P^T in the rope chunk (group 3), group 3 goes back only after the last
              // PV M-chunk has read P^T
              if (!kPInStage || m == 2) umma_commit(smem_u32(&bar_kv_empty[sb][m]));
            }
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              wait_or_flag(smem_u32(&bar_vt_full[sb][m]), (b >> 1) & 1, abort, lim);
              tc_fence_after();
#pragma unroll
              for (int ks = 0; ks < kBlockN / 16; ++ks)
                umma_ts(tmem + kTmemO + 64 * m, tmem + kTmemVT + 64 * sb + 32 * m + 8 * ks,
                        b0 + ((ks * 32) >> 4), idesc_pv_ts, (!first || ks > 0) ? 1u : 0u);
              umma_commit(smem_u32(&bar_vt_free[sb][m]));   // V^T buffer sb, chunk m reusable
            }
            if constexpr (kPInStage) umma_commit(smem_u32(&bar_kv_empty[sb][3]));
            umma_commit(smem_u32(&bar_o_done[sb]));
            SMLA_TRACE_EVENT(b, kTrSent);
          }
        }
        umma_commit(smem_u32(&bar_final_pv));
        wait_drain(smem_u32(&bar_final_pv), 0, lim);
      }
      __syncwarp();
    }
  }

  // ---- teardown: every tcgen05 op has completed (each item's epilogue waited on its last PV
  // commit, which tracks all earlier MMAs), so TMEM can be released.
  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------ split-KV merge
// One CTA per item (token, 64-head group): the n_split partial results of its slot ranges are
// merged with the standard log-sum-exp weights.  With M = max_s m_s (log2 units),
//   L = sum_s 2^(m_s - M) l_s,   O = sum_s 2^(m_s - M) O_s / (L + [sink] 2^(sink log2e - M)),
//   lse = (M + log2 L) ln 2 (sink excluded),   max_logits = max_s max_s,
// and a head without any counted slot gets O = 0, lse = +inf, max_logits = -inf.  With one
// range this is the same arithmetic as the single-pass epilogue.
constexpr int kMaxSplit = 64;
constexpr int kMaxHostChunks = 64;      // row chunks of the host-buffer entry point
constexpr int kMergeHeads = 1;       // heads per merge CTA (many small CTAs: loads in flight)
constexpr int kMergeThreads = 128;   // four value columns d per thread (float4)

__global__ void __launch_bounds__(kMergeThreads)
    splitkv_merge_kernel(const FwdParams p) {
  // grid: (item, group of kMergeHeads heads)
  __shared__ float w[kMergeHeads][kMaxSplit];
  __shared__ float sst[3][kMaxSplit][kMergeHeads];   // m, l, max of this CTA's heads per range
  __shared__ float inv[kMergeHeads];
  const int64_t item = blockIdx.x;
  const int h0 = blockIdx.y * kMergeHeads;
  const int64_t t = item / p.n_groups;
  const int g = static_cast<int>(item % p.n_groups);
  const int tid = threadIdx.x;
  const int ns = p.n_split;
  const float* st0 = p.part_stats + item * ns * (3 * kGroupHeads);
  // every statistic of every range in one parallel pass (their load latencies overlap)
  for (int e = tid; e < 3 * ns * kMergeHeads; e += kMergeThreads) {
    const int k = e / (ns * kMergeHeads), r = e % (ns * kMergeHeads);
    const int s2 = r / kMergeHeads, hh = r % kMergeHeads;
    sst[k][s2][hh] = st0[s2 * (3 * kGroupHeads) + k * kGroupHeads + h0 + hh];
  }
  __syncthreads();
  if (tid < kMergeHeads) {
    const int h = h0 + tid;
    float M = -INFINITY, mx = -INFINITY;
    for (int s2 = 0; s2 < ns; ++s2) {
      M = fmaxf(M, sst[0][s2][tid]);
      mx = fmaxf(mx, sst[2][s2][tid]);
    }
    float L = 0.f;
    for (int s2 = 0; s2 < ns; ++s2) {
      const float ms = sst[0][s2][tid];
      const float ws = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      w[tid][s2] = ws;
      L = fmaf(ws, sst[1][s2][tid], L);
    }
    const int head = g * kGroupHeads + h;
    const bool empty = !(L > 0.f);
    float den = L;
    if (p.attn_sink && !empty) den += exp2f(fmaf(__ldg(p.attn_sink + head), kLog2e, -M));
    inv[tid] = empty ? 0.f : 1.f / den;
    const int64_t o = t * p.h_q + head;
    p.lse[o] = empty ? INFINITY : (M + log2f(L)) * kLn2;
    p.max_logits[o] = empty ? -INFINITY : mx;
  }
  __syncthreads();
  const float* po = p.part_o + item * ns * static_cast<int64_t>(kGroupHeads * kDv);
  __nv_bfloat16* out_t = p.out + (t * p.h_q + g * kGroupHeads) * static_cast<int64_t>(kDv);
#pragma unroll
  for (int hh = 0; hh < kMergeHeads; ++hh) {
    const int h = h0 + hh;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s2 = 0; s2 < ns; ++s2) {
      const float ws = w[hh][s2];
      const float4 v = __ldg(reinterpret_cast<const float4*>(po + (s2 * kGroupHeads + h) * static_cast<int64_t>(kDv)) + tid);
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    const float iv = inv[hh];
    __nv_bfloat162 lo = __floats2bfloat162_rn(iv == 0.f ? 0.f : acc.x * iv, iv == 0.f ? 0.f : acc.y * iv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(iv == 0.f ? 0.f : acc.z * iv, iv == 0.f ? 0.f : acc.w * iv);
    // two 4-byte stores: out is only required to be 4-byte aligned
    uint32_t* dst = reinterpret_cast<uint32_t*>(out_t + h * kDv + 4 * tid);
    dst[0] = *reinterpret_cast<uint32_t*>(&lo);
    dst[1] = *reinterpret_cast<uint32_t*>(&hi);
  }
}

// ------------------------------------------------------------------------ wait self-test
// Runs the bounded mbarrier wait every role of the forward uses on a barrier that nothing will
// ever complete: the wait gives up after limit_ns, the kernel records SMLA_ERR_DEVICE_TIMEOUT
// in the status word and returns.  No copies, MMAs or tensor memory are involved.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  wait_or_flag(smem_u32(&bar), 0, &abort_flag, limit_ns);
}

// ------------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle, box = box_cols
// x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  std::memset(m, 0, sizeof(*m));
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int D_QK, bool DYNAMIC, bool PAGED, bool SPLIT>
smla_status launch_one(const CUtensorMap& qm, const CUtensorMap& kvm, const FwdParams& p,
                       cudaStream_t stream) {
  auto kern = sparse_mla_fwd_kernel<D_QK, DYNAMIC, PAGED, SPLIT>;
  constexpr int kChunks = D_QK / 64;
  const size_t smem = 3 * kChunks * 8192 + (kChunks > 8 ? 0 : 2 * 8192) + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return SMLA_ERR_LAUNCH;
  // persistent: one CTA per SM (the shared-memory footprint admits only one), work units
  // assigned round-robin
  const int sms = sm_count();
  if (sms <= 0) return SMLA_ERR_LAUNCH;
  const int64_t units = SPLIT ? p.n_items * p.n_split : p.n_items;
  const int64_t grid = units < sms ? units : sms;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(qm, kvm, p);
  if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_LAUNCH;
  if constexpr (SPLIT) {
    splitkv_merge_kernel<<<dim3(static_cast<unsigned>(p.n_items), kGroupHeads / kMergeHeads), kMergeThreads, 0,
                           stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_LAUNCH;
  }
  return SMLA_OK;
}

template <bool PAGED>
smla_status dispatch(int d_qk, bool dynamic, const CUtensorMap& qm, const CUtensorMap& kvm,
                     const FwdParams& p, cudaStream_t stream) {
  // topk_length presence is a compile-time choice (FlashMLA PR #216, "Why template<bool
  // DYNAMIC_TOPK>"): the fixed path carries no length load or tail predicate.
  const bool split = p.n_split > 1;
  if (d_qk == 512) {
    if (split)
      return dynamic ? launch_one<512, true, PAGED, true>(qm, kvm, p, stream)
                     : launch_one<512, false, PAGED, true>(qm, kvm, p, stream);
    return dynamic ? launch_one<512, true, PAGED, false>(qm, kvm, p, stream)
                   : launch_one<512, false, PAGED, false>(qm, kvm, p, stream);
  }
  if (split)
    return dynamic ? launch_one<576, true, PAGED, true>(qm, kvm, p, stream)
                   : launch_one<576, false, PAGED, true>(qm, kvm, p, stream);
  return dynamic ? launch_one<576, true, PAGED, false>(qm, kvm, p, stream)
                 : launch_one<576, false, PAGED, false>(qm, kvm, p, stream);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

smla_status check_common(const void* q, const void* kv, const int32_t* indices, const void* out,
                         const float* lse, const float* max_logits, int64_t s_q, int h_q,
                         int d_qk, int d_v, int topk, float sm_scale) {
  if (s_q < 0 || h_q <= 0 || h_q % kGroupHeads != 0 || h_q > 1024) return SMLA_ERR_BAD_SHAPE;
  if (d_qk != 512 && d_qk != 576) return SMLA_ERR_BAD_SHAPE;
  if (d_v != kDv || d_v > d_qk) return SMLA_ERR_BAD_SHAPE;
  if (topk < 1) return SMLA_ERR_BAD_SHAPE;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return SMLA_ERR_BAD_SHAPE;
  if (s_q * static_cast<int64_t>(h_q) > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
  if (s_q == 0) return SMLA_OK;
  if (!q || !kv || !indices || !out || !lse || !max_logits) return SMLA_ERR_NULL_PTR;
  if (!aligned16(q) || !aligned16(kv) || !aligned4(indices) || !aligned4(out) || !aligned4(lse) ||
      !aligned4(max_logits))
    return SMLA_ERR_MISALIGNED;
  return SMLA_OK;
}

// the backward kernel and its host side share the helpers above
#include "sparse_mla_bwd.cuh"

}  // namespace
}  // namespace smla


namespace smla {
namespace {

// Bytes of split-KV workspace for s_q rows x (h_q / 64) groups x n_split ranges: the partial
// O block of every unit, then its statistics (256-byte aligned).
size_t splitkv_bytes(int64_t s_q, int h_q, int n_split, size_t* stats_offset) {
  const int64_t units = s_q * (h_q / kGroupHeads) * n_split;
  const size_t o_bytes = static_cast<size_t>(units) * kGroupHeads * kDv * sizeof(float);
  const size_t off = (o_bytes + 255) & ~static_cast<size_t>(255);
  if (stats_offset) *stats_offset = off;
  return off + static_cast<size_t>(units) * 3 * kGroupHeads * sizeof(float);
}

// Validates the split-KV arguments and points p at the workspace.  n_split == 1 needs none.
smla_status set_split(FwdParams& p, int64_t s_q, int h_q, int n_split, void* workspace,
                      size_t workspace_bytes) {
  if (n_split < 1 || n_split > kMaxSplit) return SMLA_ERR_BAD_SHAPE;
  if (s_q * (h_q / kGroupHeads) * static_cast<int64_t>(n_split) > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
  p.n_split = n_split;
  // one range needs no workspace; with no rows nothing runs and no pointer is inspected
  if (n_split == 1 || s_q == 0) return SMLA_OK;
  if (!workspace) return SMLA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SMLA_ERR_MISALIGNED;
  size_t stats_off = 0;
  if (workspace_bytes < splitkv_bytes(s_q, h_q, n_split, &stats_off)) return SMLA_ERR_WORKSPACE;
  p.part_o = static_cast<float*>(workspace);
  p.part_stats = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + stats_off);
  return SMLA_OK;
}

smla_status fwd_flat(const void* q, const void* kv, const int32_t* indices, const int32_t* topk_length,
                     const float* attn_sink, float sm_scale, int d_v, void* out, float* lse,
                     float* max_logits, int64_t s_q, int64_t s_kv, int h_q, int d_qk, int topk,
                     int n_split, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (s_kv < 0 || s_kv > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
  // with an empty KV every slot is invalid and kv is never read: it may then be NULL
  const void* kv_base = s_kv > 0 ? kv : q;
  smla_status st = check_common(q, kv_base, indices, out, lse, max_logits, s_q, h_q, d_qk, d_v,
                                topk, sm_scale);
  if (st != SMLA_OK) return st;
  FwdParams p{};
  st = set_split(p, s_q, h_q, n_split, workspace, workspace_bytes);
  if (st != SMLA_OK || s_q == 0) return st;
  if (attn_sink && !aligned4(attn_sink)) return SMLA_ERR_MISALIGNED;
  if (topk_length && !aligned4(topk_length)) return SMLA_ERR_MISALIGNED;
  CUtensorMap qm, kvm;
  if (!make_map(&qm, q, static_cast<uint64_t>(s_q) * h_q, d_qk, 64)) return SMLA_ERR_TENSOR_MAP;
  // an empty KV still needs a one-row map; every slot is then invalid and never read
  if (!make_map(&kvm, kv_base, s_kv > 0 ? static_cast<uint64_t>(s_kv) : 1u, d_qk, 1))
    return SMLA_ERR_TENSOR_MAP;
  p.indices = indices;
  p.topk_length = topk_length;
  p.attn_sink = attn_sink;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.max_logits = max_logits;
  p.sm_scale = sm_scale;
  p.s_q = s_q;
  p.s_kv = s_kv;
  p.h_q = h_q;
  p.topk = topk;
  p.n_groups = h_q / kGroupHeads;
  p.n_items = s_q * p.n_groups;
  p.s_q_per_req = 1;
  p.page_block = 1;
  p.max_blocks = 1;
  p.pool_rows = s_kv;
  return dispatch<false>(d_qk, topk_length != nullptr, qm, kvm, p, stream);
}

smla_status fwd_paged(const void* q, const void* kv_pool, int64_t pool_rows, const int32_t* block_table,
                      int max_blocks, int page_block, const int32_t* seqlens_k, int64_t s_kv_per_req,
                      int s_q_per_req, const int32_t* indices, const int32_t* topk_length,
                      const float* attn_sink, float sm_scale, int d_v, void* out, float* lse,
                      float* max_logits, int64_t s_q, int h_q, int d_qk, int topk, int n_split,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  smla_status st = check_common(q, kv_pool, indices, out, lse, max_logits, s_q, h_q, d_qk, d_v,
                                topk, sm_scale);
  if (st != SMLA_OK) return st;
  FwdParams p{};
  st = set_split(p, s_q, h_q, n_split, workspace, workspace_bytes);
  if (st != SMLA_OK || s_q == 0) return st;
  if (pool_rows < 1 || pool_rows > INT32_MAX || max_blocks < 1 || page_block < 1 ||
      s_q_per_req < 1 || s_kv_per_req < 0 || s_kv_per_req > INT32_MAX ||
      static_cast<int64_t>(max_blocks) * page_block > INT32_MAX || s_q % s_q_per_req != 0)
    return SMLA_ERR_BAD_SHAPE;
  if (!block_table) return SMLA_ERR_NULL_PTR;
  if (!aligned4(block_table) || (seqlens_k && !aligned4(seqlens_k)) ||
      (attn_sink && !aligned4(attn_sink)) || (topk_length && !aligned4(topk_length)))
    return SMLA_ERR_MISALIGNED;
  CUtensorMap qm, kvm;
  if (!make_map(&qm, q, static_cast<uint64_t>(s_q) * h_q, d_qk, 64)) return SMLA_ERR_TENSOR_MAP;
  if (!make_map(&kvm, kv_pool, static_cast<uint64_t>(pool_rows), d_qk, 1)) return SMLA_ERR_TENSOR_MAP;
  p.indices = indices;
  p.topk_length = topk_length;
  p.attn_sink = attn_sink;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.max_logits = max_logits;
  p.sm_scale = sm_scale;
  p.s_q = s_q;
  p.s_kv = s_kv_per_req;
  p.h_q = h_q;
  p.topk = topk;
  p.n_groups = h_q / kGroupHeads;
  p.n_items = s_q * p.n_groups;
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.max_blocks = max_blocks;
  p.page_block = page_block;
  p.s_q_per_req = s_q_per_req;
  p.pool_rows = pool_rows;
  return dispatch<true>(d_qk, topk_length != nullptr, qm, kvm, p, stream);
}

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" {

smla_status sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices,
                           const int32_t* topk_length, const float* attn_sink, float sm_scale,
                           int d_v, void* out, float* lse, float* max_logits, int64_t s_q,
                           int64_t s_kv, int h_q, int d_qk, int topk, cudaStream_t stream) {
  return fwd_flat(q, kv, indices, topk_length, attn_sink, sm_scale, d_v, out, lse, max_logits, s_q,
                  s_kv, h_q, d_qk, topk, 1, nullptr, 0, stream);
}

smla_status sparse_mla_fwd_paged(const void* q, const void* kv_pool, int64_t pool_rows,
                                 const int32_t* block_table, int max_blocks, int page_block,
                                 const int32_t* seqlens_k, int64_t s_kv_per_req, int s_q_per_req,
                                 const int32_t* indices, const int32_t* topk_length,
                                 const float* attn_sink, float sm_scale, int d_v, void* out,
                                 float* lse, float* max_logits, int64_t s_q, int h_q, int d_qk,
                                 int topk, cudaStream_t stream) {
  return fwd_paged(q, kv_pool, pool_rows, block_table, max_blocks, page_block, seqlens_k, s_kv_per_req,
                   s_q_per_req, indices, topk_length, attn_sink, sm_scale, d_v, out, lse, max_logits,
                   s_q, h_q, d_qk, topk, 1, nullptr, 0, stream);
}

smla_status sparse_mla_fwd_paged_splitkv_static(
    const void* q, const void* kv_pool, int64_t pool_rows, const int32_t* block_table, int max_blocks,
    int page_block, const int32_t* seqlens_k, int64_t s_kv_per_req, int s_q_per_req,
    const int32_t* indices, const int32_t* topk_length, const float* attn_sink, float sm_scale, int d_v,
    void* out, float* lse, float* max_logits, int64_t s_q, int h_q, int d_qk, int topk, int n_split,
    cudaStream_t stream) {
  // the scratch is fixed: larger problems are rejected before anything runs
  if (s_q >= 0 && h_q > 0 && h_q % kGroupHeads == 0 && n_split > 1 && n_split <= kMaxSplit &&
      splitkv_bytes(s_q, h_q, n_split, nullptr) > kStaticScratchBytes)
    return SMLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (n_split > 1 && s_q > 0) {
    // the scratch's address on the current device, looked up once per device with that device
    // current (each device has its own copy of the array)
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SMLA_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] && cudaGetSymbolAddress(&addr[dev], g_splitkv_scratch) != cudaSuccess) {
      addr[dev] = nullptr;
      return SMLA_ERR_LAUNCH;
    }
    scratch = addr[dev];
  }
  return fwd_paged(q, kv_pool, pool_rows, block_table, max_blocks, page_block, seqlens_k, s_kv_per_req,
                   s_q_per_req, indices, topk_length, attn_sink, sm_scale, d_v, out, lse, max_logits,
                   s_q, h_q, d_qk, topk, n_split, scratch, kStaticScratchBytes, stream);
}

smla_status sparse_mla_fwd_host(const void* q_host, const void* kv_host, const int32_t* indices_host,
                                const int32_t* topk_length_host, const float* attn_sink_host, float sm_scale,
                                int d_v, void* out_host, float* lse_host, float* max_logits_host, int64_t s_q,
                                int64_t s_kv, int h_q, int d_qk, int topk, void* q_dev, void* kv_dev,
                                int32_t* indices_dev, int32_t* topk_length_dev, float* attn_sink_dev, void* out_dev,
                                float* lse_dev, float* max_logits_dev, int n_chunks, cudaStream_t stream,
                                cudaStream_t copy_in, cudaStream_t copy_out) {
  // every argument is checked before anything is enqueued
  if (n_chunks < 1 || n_chunks > kMaxHostChunks) return SMLA_ERR_BAD_SHAPE;
  if (s_kv < 0 || s_kv > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
  smla_status st = check_common(q_dev, s_kv > 0 ? kv_dev : q_dev, indices_dev, out_dev, lse_dev, max_logits_dev,
                                s_q, h_q, d_qk, d_v, topk, sm_scale);
  if (st != SMLA_OK || s_q == 0) return st;
  if (!q_host || !indices_host || !out_host || !lse_host || !max_logits_host || (s_kv > 0 && !kv_host))
    return SMLA_ERR_NULL_PTR;
  if ((topk_length_host == nullptr) != (topk_length_dev == nullptr) ||
      (attn_sink_host == nullptr) != (attn_sink_dev == nullptr))
    return SMLA_ERR_NULL_PTR;
  if ((attn_sink_dev && !aligned4(attn_sink_dev)) || (topk_length_dev && !aligned4(topk_length_dev)))
    return SMLA_ERR_MISALIGNED;
  const int64_t rows_per = (s_q + n_chunks - 1) / n_chunks;
  const int chunks = static_cast<int>((s_q + rows_per - 1) / rows_per);
  // Events order the three streams: inputs of chunk i -> its kernel -> its outputs.  They come
  // from a pool per device, created on the first call there; re-recording an event is safe for
  // the waits enqueued earlier, and the lock keeps two host threads from recording the same
  // events at once while they enqueue.
  constexpr int kEvents = 2 * kMaxHostChunks + 3;
  static std::mutex pool_mu;
  static cudaEvent_t pool[64][kEvents];
  static bool pool_ready[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SMLA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(pool_mu);
  if (!pool_ready[dev]) {
    for (int e = 0; e < kEvents; ++e) {
      if (cudaEventCreateWithFlags(&pool[dev][e], cudaEventDisableTiming) != cudaSuccess) {
        for (int k = 0; k < e; ++k) cudaEventDestroy(pool[dev][k]);
        return SMLA_ERR_LAUNCH;
      }
    }
    pool_ready[dev] = true;
  }
  cudaEvent_t* ev = pool[dev];
  cudaEvent_t ev_kv = ev[0], ev_done = ev[1], ev_start = ev[2];
  auto ev_in = [&](int i) { return ev[3 + 2 * i]; };
  auto ev_k = [&](int i) { return ev[4 + 2 * i]; };
  const size_t q_row = static_cast<size_t>(h_q) * d_qk * 2, o_row = static_cast<size_t>(h_q) * d_v * 2;
  const size_t s_row = static_cast<size_t>(h_q) * sizeof(float), i_row = static_cast<size_t>(topk) * 4;
  auto h2d = [&](void* dst, const void* src, size_t n) {
    return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, copy_in) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t n) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, copy_out) == cudaSuccess;
  };
  // the copies come after the work already queued on `stream` (which may still read the
  // device buffers), as if the whole call ran on `stream`
  bool ok = cudaEventRecord(ev_start, stream) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(copy_in, ev_start, 0) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(copy_out, ev_start, 0) == cudaSuccess;
  // the inputs every chunk shares, then each chunk's rows
  ok = ok && h2d(kv_dev, kv_host, static_cast<size_t>(s_kv) * d_qk * 2);
  if (attn_sink_dev) ok = ok && h2d(attn_sink_dev, attn_sink_host, s_row);
  ok = ok && cudaEventRecord(ev_kv, copy_in) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(stream, ev_kv, 0) == cudaSuccess;
  for (int i = 0; i < chunks && ok && st == SMLA_OK; ++i) {
    const int64_t r0 = i * rows_per, n = std::min(rows_per, s_q - r0);
    ok = ok && h2d(static_cast<uint8_t*>(q_dev) + r0 * q_row, static_cast<const uint8_t*>(q_host) + r0 * q_row,
                   n * q_row);
    ok = ok && h2d(indices_dev + r0 * topk, indices_host + r0 * topk, n * i_row);
    if (topk_length_dev) ok = ok && h2d(topk_length_dev + r0, topk_length_host + r0, n * 4);
    ok = ok && cudaEventRecord(ev_in(i), copy_in) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(stream, ev_in(i), 0) == cudaSuccess;
    if (!ok) break;
    // the rows of one chunk are an independent forward call: the same bits as one call on all
    st = fwd_flat(static_cast<uint8_t*>(q_dev) + r0 * q_row, kv_dev, indices_dev + r0 * topk,
                  topk_length_dev ? topk_length_dev + r0 : nullptr, attn_sink_dev, sm_scale, d_v,
                  static_cast<uint8_t*>(out_dev) + r0 * o_row, lse_dev + r0 * h_q, max_logits_dev + r0 * h_q, n,
                  s_kv, h_q, d_qk, topk, 1, nullptr, 0, stream);
    ok = ok && cudaEventRecord(ev_k(i), stream) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(copy_out, ev_k(i), 0) == cudaSuccess;
    ok = ok && d2h(static_cast<uint8_t*>(out_host) + r0 * o_row, static_cast<const uint8_t*>(out_dev) + r0 * o_row,
                   n * o_row);
    ok = ok && d2h(lse_host + r0 * h_q, lse_dev + r0 * h_q, n * s_row);
    ok = ok && d2h(max_logits_host + r0 * h_q, max_logits_dev + r0 * h_q, n * s_row);
  }
  // the caller's stream completes only after the last copy out
  ok = ok && cudaEventRecord(ev_done, copy_out) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(stream, ev_done, 0) == cudaSuccess;
  if (st != SMLA_OK) return st;
  return ok ? SMLA_OK : SMLA_ERR_LAUNCH;
}

smla_status sparse_mla_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > kDefaultWaitLimitNs) return SMLA_ERR_BAD_SHAPE;
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_LAUNCH;
}

size_t sparse_mla_splitkv_workspace_size(int64_t s_q, int h_q, int n_split) {
  if (s_q < 0 || h_q <= 0 || h_q % kGroupHeads != 0 || n_split < 1 || n_split > kMaxSplit) return 0;
  if (n_split == 1) return 0;
  return splitkv_bytes(s_q, h_q, n_split, nullptr);
}

smla_status sparse_mla_fwd_splitkv(const void* q, const void* kv, const int32_t* indices,
                                   const int32_t* topk_length, const float* attn_sink, float sm_scale,
                                   int d_v, void* out, float* lse, float* max_logits, int64_t s_q,
                                   int64_t s_kv, int h_q, int d_qk, int topk, int n_split,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fwd_flat(q, kv, indices, topk_length, attn_sink, sm_scale, d_v, out, lse, max_logits, s_q,
                  s_kv, h_q, d_qk, topk, n_split, workspace, workspace_bytes, stream);
}

smla_status sparse_mla_fwd_paged_splitkv(const void* q, const void* kv_pool, int64_t pool_rows,
                                         const int32_t* block_table, int max_blocks, int page_block,
                                         const int32_t* seqlens_k, int64_t s_kv_per_req,
                                         int s_q_per_req, const int32_t* indices,
                                         const int32_t* topk_length, const float* attn_sink,
                                         float sm_scale, int d_v, void* out, float* lse,
                                         float* max_logits, int64_t s_q, int h_q, int d_qk, int topk,
                                         int n_split, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
  return fwd_paged(q, kv_pool, pool_rows, block_table, max_blocks, page_block, seqlens_k, s_kv_per_req,
                   s_q_per_req, indices, topk_length, attn_sink, sm_scale, d_v, out, lse, max_logits,
                   s_q, h_q, d_qk, topk, n_split, workspace, workspace_bytes, stream);
}

smla_status sparse_mla_device_status(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return SMLA_ERR_LAUNCH;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_device_status, &z, sizeof(int)) != cudaSuccess) return SMLA_ERR_LAUNCH;
  }
  return static_cast<smla_status>(v);
}

const char* sparse_mla_status_string(smla_status s) {
  switch (s) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_NULL_PTR: return "null pointer argument";
    case SMLA_ERR_BAD_SHAPE: return "unsupported shape or argument value";
    case SMLA_ERR_MISALIGNED: return "misaligned pointer";
    case SMLA_ERR_LAUNCH: return "kernel launch failed";
    case SMLA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case SMLA_ERR_TENSOR_MAP: return "TMA descriptor encoding failed";
    case SMLA_ERR_WORKSPACE: return "split-KV workspace missing or too small";
  }
  return "unknown status";
}

int sparse_mla_abi_version(void) { return SMLA_ABI_VERSION; }

smla_status sparse_mla_bwd(const void* q, const void* kv, const void* out, const void* dout,
                           const int32_t* indices, const int32_t* topk_length, const float* attn_sink,
                           const float* lse, float sm_scale, int d_v, float* dq, float* dkv, float* dsink,
                           int64_t s_q, int64_t s_kv, int h_q, int d_qk, int topk, smla_stream_t stream) {
  return smla::bwd_flat(q, kv, out, dout, indices, topk_length, attn_sink, lse, sm_scale, d_v, dq, dkv, dsink,
                        s_q, s_kv, h_q, d_qk, topk, reinterpret_cast<cudaStream_t>(stream));
}

#ifdef SMLA_TRACE
// Debug builds only: copies the pipeline trace of CTA 0 ([256 blocks][12 events] int64 clock
// stamps) into `dst` (host memory).
int sparse_mla_trace_fetch(long long* dst) {
  return cudaMemcpyFromSymbol(dst, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -1;
}
#endif

}  // extern "C"
