// Sparse MLA attention forward (DSA top-k) for sm_103a.
//
// Each query token t attends to its own list of top-k slots into one shared latent KV
// (h_kv = 1; K = kv[:, :d_qk], V = kv[:, :d_v]).  A slot j counts iff j < L_t and
// 0 <= idx[t][j] < s_kv, where L_t is the row's effective length: the caller's topk_length[t]
// clamped to [0, topk], or, when no topk_length is given, one past the last valid slot found
// by a tail scan in the prologue (FlashMLA PR #196, "Fix").  Rows with no valid slot return
// O = 0, lse = +inf, max_logits = -inf (FlashMLA PR #196, "Correctness notes").  The optional
// per-head attention sink is a value-less virtual key in the softmax denominator (FlashMLA
// PR #198, "Summary" item 2).
//
// One CTA computes one (token, group of 64 heads).  Warp roles (288 threads):
//   warps 0-3  producer : TMA gather4 of the selected KV rows into a 2-stage ring; slots that
//                         are invalid or past L_t get an out-of-range row coordinate, so TMA
//                         zero-fills them and their index is never used as an address
//   warps 4-7  softmax  : online exp2 softmax on S (one head per TMEM lane), P -> smem,
//                         lazy O rescale, epilogue (sink, normalise, write O / lse / max)
//   warp  8    MMA      : TMEM allocation and tcgen05.mma issue (one elected thread)
// Tensor-core work per 64-key block:
//   S[64 heads x 64 keys]  = Q_g . K_blk^T        (M=64, N=64,  K=d_qk; both K-major SW128)
//   O^T[512 x 64 heads]   += V_blk^T . P^T        (4 x M=128, N=64, K=64; V^T read MN-major
//                                                  straight out of the gathered K block)
// TMEM: O^T in columns [0,256), S double buffer in [256,384).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kBlockN = 64;            // keys per k-block
constexpr int kGroupHeads = 64;        // heads per CTA
constexpr int kDv = 512;               // value width (first d_v columns of each kv row)
constexpr int kThreads = 288;
constexpr int kProducerThreads = 128;  // warps 0-3
static_assert(kProducerThreads == 32 * 4, "producer warps precede the softmax warps");
constexpr int kSoftmaxWarp0 = 4;       // warps 4-7
constexpr int kMmaWarp = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;         // O^T: 4 chunks x 64 columns
constexpr uint32_t kTmemS = 256;       // S buffers: 256 + 64*b
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;   // rescale O only when the running max grows by > 2^8

__device__ int g_device_status = 0;    // SMLA_ERR_DEVICE_TIMEOUT once any wait gave up

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
  // paged KV cache
  const int32_t* block_table;  // [n_req, max_blocks]
  const int32_t* seqlens_k;    // [n_req] or null
  int max_blocks;
  int page_block;
  int s_q_per_req;
  int64_t pool_rows;           // rows the KV tensor map covers
  uint64_t wait_limit_ns;
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

template <int D_QK, bool DYNAMIC, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_fwd_kernel(const __grid_constant__ CUtensorMap q_map,
                          const __grid_constant__ CUtensorMap kv_map, const FwdParams p) {
  constexpr int kChunks = D_QK / 64;                 // 128-byte column chunks of a row
  constexpr uint32_t kTileBytes = kChunks * 8192u;   // 64 rows x D_QK bf16 (= Q tile = stage)
  constexpr int kQkSteps = D_QK / 16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kTileBytes;                  // stage s at sKV + s * kTileBytes
  uint8_t* sP = smem + 3 * kTileBytes;               // P as [64 heads][64 keys] bf16, SW128

  __shared__ __align__(8) uint64_t bar_q, bar_full[2], bar_empty[2], bar_s[2], bar_p, bar_o;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int s_last;
  __shared__ float s_alpha[kGroupHeads];
  __shared__ float s_inv[kGroupHeads];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) / p.n_groups;
  const int g = static_cast<int>(static_cast<int64_t>(blockIdx.x) % p.n_groups);
  const int topk = p.topk;
  const int32_t* idx_row = p.indices + t * static_cast<int64_t>(topk);
  const int64_t kv_len = row_kv_len<PAGED>(p, t);
  volatile int* abort = &abort_flag;

  // ---- prologue, part 1: issue the effective-length loads before any setup, so they are in
  // flight while barriers are initialised, Q is requested and TMEM is allocated.
  int my_last = -1;
  int given_len = 0;
  if (DYNAMIC) {
    if (tid == 0) given_len = __ldg(p.topk_length + t);
  } else {
    for (int j = tid; j < topk; j += kThreads) {
      const int v = __ldg(idx_row + j);
      if (slot_ok<PAGED>(p, v, kv_len)) my_last = j;
    }
  }

  if (tid == 0) {
    abort_flag = 0;
    s_last = -1;
    mbar_init(smem_u32(&bar_q), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
      mbar_init(smem_u32(&bar_s[s]), 1);
    }
    mbar_init(smem_u32(&bar_p), 128);
    mbar_init(smem_u32(&bar_o), 1);
    fence_mbar_init();
    // Q tile of this (token, head group): 64 rows of the [s_q*h_q, d_qk] view.
    mbar_arrive_expect_tx(smem_u32(&bar_q), kTileBytes);
    const int qrow = static_cast<int>(t * p.h_q + g * kGroupHeads);
    for (int c = 0; c < kChunks; ++c)
      tma_load_2d(smem_u32(sQ + c * 8192), &q_map, 64 * c, qrow, smem_u32(&bar_q));
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- prologue, part 2: consume.  Every warp then derives the same loop bound from the same
  // value, so the k-block loop is uniform across all roles.
  if (DYNAMIC) {
    if (tid == 0) s_last = min(max(given_len, 0), topk) - 1;
  } else {
    int m = my_last;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && m >= 0) atomicMax(&s_last, m);
  }
  __syncthreads();
  const int L = s_last + 1;
  const int nblk = max((L + kBlockN - 1) / kBlockN, 1);
  const uint32_t tmem = tmem_slot;

  if (warp < kSoftmaxWarp0) {
    // ======================================================== producer: TMA gather
    const int pi = tid;                 // 0..127
    const int grp = pi & 15;            // 4-row group within the block
    const int c0 = pi >> 4;             // column chunk 0..7
    for (int k = 0; k < nblk; ++k) {
      const int s = k & 1;
      if (k >= 2) wait_or_flag(smem_u32(&bar_empty[s]), ((k >> 1) - 1) & 1, abort, p.wait_limit_ns);
      if (pi == 0) mbar_arrive_expect_tx(smem_u32(&bar_full[s]), kTileBytes);
      int rows[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = k * kBlockN + grp * 4 + i;
        int coord = -1;                 // out of range: zero-filled, never read
        if (j < L) {
          const int v = __ldg(idx_row + j);
          if (slot_ok<PAGED>(p, v, kv_len)) coord = kv_row_of<PAGED>(p, t, v);
        }
        rows[i] = coord;
      }
      uint8_t* st = sKV + s * kTileBytes;
      const uint32_t bar = smem_u32(&bar_full[s]);
      tma_gather4(smem_u32(st + c0 * 8192 + grp * 512), &kv_map, 64 * c0, rows[0], rows[1], rows[2],
                  rows[3], bar);
      if (kChunks > 8 && pi < 16 * (kChunks - 8)) {
        const int c1 = 8 + (pi >> 4);
        tma_gather4(smem_u32(st + c1 * 8192 + grp * 512), &kv_map, 64 * c1, rows[0], rows[1],
                    rows[2], rows[3], bar);
      }
    }
  } else if (warp < kMmaWarp) {
    // ======================================================== softmax / correction / epilogue
    const int q = warp - kSoftmaxWarp0;          // TMEM lane quadrant 0..3
    const bool row_owner = lane < 16;            // M=64 layout: heads live in lanes 0-15
    const int h = 16 * q + lane;                 // local head (valid when row_owner)
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const float c = p.sm_scale * kLog2e;
    float m_used = -INFINITY;                    // running exponent offset (log2 units)
    float s_max = -INFINITY;                     // running max of raw q.k
    float l_sum = 0.f;

    for (int k = 0; k < nblk; ++k) {
      const int b = k & 1;
      // validity of the block's 64 slots, from the indices (never from the gathered data)
      const int ja = k * kBlockN + 2 * lane, jb = ja + 1;
      bool oka = false, okb = false;
      if (ja < L) oka = slot_ok<PAGED>(p, __ldg(idx_row + ja), kv_len);
      if (jb < L) okb = slot_ok<PAGED>(p, __ldg(idx_row + jb), kv_len);
      const uint32_t even_bits = __ballot_sync(0xffffffffu, oka);
      const uint32_t odd_bits = __ballot_sync(0xffffffffu, okb);

      wait_or_flag(smem_u32(&bar_s[b]), (k >> 1) & 1, abort, p.wait_limit_ns);
      tc_fence_after();
      float sv[kBlockN];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + kTmemS + 64 * b + 16 * i, r);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sv[16 * i + jj] = __uint_as_float(r[jj]);
      }
      tmem_ld_wait();

      float alpha = 1.f;
      bool need_rescale = false;
      uint32_t pk[kBlockN / 2];
      if (row_owner) {
        float bm = -INFINITY;
#pragma unroll
        for (int j = 0; j < kBlockN; ++j) {
          const bool ok = ((((j & 1) ? odd_bits : even_bits) >> (j >> 1)) & 1u) != 0u;
          sv[j] = ok ? sv[j] : -INFINITY;
          bm = fmaxf(bm, sv[j]);
        }
        s_max = fmaxf(s_max, bm);
        const float bm2 = bm * c;
        if (bm2 > m_used + kRescaleLog2) {
          alpha = fast_exp2(m_used - bm2);       // 0 when m_used was -inf
          m_used = bm2;
          need_rescale = true;
        }
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < kBlockN; j += 2) {
          const float p0 = (sv[j] == -INFINITY) ? 0.f : fast_exp2(fmaf(sv[j], c, -m_used));
          const float p1 = (sv[j + 1] == -INFINITY) ? 0.f : fast_exp2(fmaf(sv[j + 1], c, -m_used));
          ls += p0 + p1;
          pk[j >> 1] = pack_bf16x2(p0, p1);
        }
        l_sum = fmaf(l_sum, alpha, ls);
      }
      // O^T must be rescaled before PV(k) only if some head's offset moved and O already
      // holds earlier blocks.
      const bool any_rescale = named_bar_or(1, 128, need_rescale && k > 0);
      // PV(k-1) must be complete before P is overwritten or O^T is touched.
      if (k > 0) wait_or_flag(smem_u32(&bar_o), (k - 1) & 1, abort, p.wait_limit_ns);
      if (any_rescale) {
        if (row_owner) s_alpha[h] = alpha;
        named_bar_sync(2, 128);
        tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t r[16];
            const uint32_t addr = tmem + lane_base + kTmemO + 64 * m + 16 * i;
            tmem_ld16(addr, r);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              r[jj] = __float_as_uint(__uint_as_float(r[jj]) * s_alpha[16 * i + jj]);
            tmem_st16(addr, r);
          }
        }
        tmem_st_wait();
        named_bar_sync(2, 128);                  // s_alpha is reused next block
      }
      if (row_owner) {
        uint8_t* row = sP + h * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          *reinterpret_cast<uint4*>(row + ((u ^ (h & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p));
    }

    // ---- epilogue
    wait_or_flag(smem_u32(&bar_o), (nblk - 1) & 1, abort, p.wait_limit_ns);
    tc_fence_after();
    const int head = g * kGroupHeads + h;
    if (row_owner) {
      const bool empty = !(l_sum > 0.f);
      float den = l_sum;
      if (p.attn_sink) den += exp2f(fmaf(__ldg(p.attn_sink + head), kLog2e, -m_used));
      s_inv[h] = empty ? 0.f : 1.f / den;
      const int64_t o = t * p.h_q + head;
      p.lse[o] = empty ? INFINITY : (m_used + log2f(l_sum)) * kLn2;
      p.max_logits[o] = empty ? -INFINITY : s_max * p.sm_scale;
    }
    named_bar_sync(2, 128);
    __nv_bfloat16* out_t = p.out + (t * p.h_q + g * kGroupHeads) * static_cast<int64_t>(kDv);
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      const int d = 128 * m + 32 * q + lane;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + kTmemO + 64 * m + 16 * i, r);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int hh = 16 * i + jj;
          const float inv = s_inv[hh];
          const float val = (inv == 0.f) ? 0.f : __uint_as_float(r[jj]) * inv;
          out_t[static_cast<int64_t>(hh) * kDv + d] = __float2bfloat16_rn(val);
        }
      }
    }
  } else {
    // ======================================================== MMA issuer
    if (lane == 0) {
      wait_or_flag(smem_u32(&bar_q), 0, abort, p.wait_limit_ns);
      tc_fence_after();
      constexpr uint32_t idesc_qk = make_idesc_bf16(64, kBlockN, false, false);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, kGroupHeads, true, false);
      const uint32_t q_base = smem_u32(sQ);
      const uint32_t kv_base = smem_u32(sKV);
      const uint32_t p_base = smem_u32(sP);
      auto issue_pv = [&](int j) {
        wait_or_flag(smem_u32(&bar_p), j & 1, abort, p.wait_limit_ns);
        tc_fence_after();
        const uint32_t st = kv_base + (j & 1) * kTileBytes;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int ks = 0; ks < kBlockN / 16; ++ks) {
            const uint64_t a = make_sdesc_sw128(st + (2 * m) * 8192 + ks * 2048, 8192, 1024);
            const uint64_t bd = make_sdesc_sw128(p_base + ks * 32, 16, 1024);
            umma_ss(tmem + kTmemO + 64 * m, a, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&bar_empty[j & 1]));
        umma_commit(smem_u32(&bar_o));
      };
      for (int k = 0; k < nblk; ++k) {
        const int s = k & 1;
        wait_or_flag(smem_u32(&bar_full[s]), (k >> 1) & 1, abort, p.wait_limit_ns);
        tc_fence_after();
        const uint32_t st = kv_base + s * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kQkSteps; ++ks) {
          const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
          umma_ss(tmem + kTmemS + 64 * s, make_sdesc_sw128(q_base + off, 16, 1024),
                  make_sdesc_sw128(st + off, 16, 1024), idesc_qk, ks > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bar_s[s]));
        if (k > 0) issue_pv(k - 1);
      }
      issue_pv(nblk - 1);
    }
    __syncwarp();
  }

  // ---- teardown: every tcgen05 op has completed (the epilogue waited on the last PV commit,
  // which tracks all earlier MMAs), so TMEM can be released.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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

template <int D_QK, bool DYNAMIC, bool PAGED>
smla_status launch_one(const CUtensorMap& qm, const CUtensorMap& kvm, const FwdParams& p,
                       cudaStream_t stream) {
  auto kern = sparse_mla_fwd_kernel<D_QK, DYNAMIC, PAGED>;
  const size_t smem = 3 * (D_QK / 64) * 8192 + 8192 + 1024;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return SMLA_ERR_LAUNCH;
  const int64_t grid = p.s_q * p.n_groups;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(qm, kvm, p);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_LAUNCH;
}

template <bool PAGED>
smla_status dispatch(int d_qk, bool dynamic, const CUtensorMap& qm, const CUtensorMap& kvm,
                     const FwdParams& p, cudaStream_t stream) {
  // topk_length presence is a compile-time choice (FlashMLA PR #216, "Why template<bool
  // DYNAMIC_TOPK>"): the fixed path carries no length load or tail predicate.
  if (d_qk == 512)
    return dynamic ? launch_one<512, true, PAGED>(qm, kvm, p, stream)
                   : launch_one<512, false, PAGED>(qm, kvm, p, stream);
  return dynamic ? launch_one<576, true, PAGED>(qm, kvm, p, stream)
                 : launch_one<576, false, PAGED>(qm, kvm, p, stream);
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

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" {

smla_status sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices,
                           const int32_t* topk_length, const float* attn_sink, float sm_scale,
                           int d_v, void* out, float* lse, float* max_logits, int64_t s_q,
                           int64_t s_kv, int h_q, int d_qk, int topk, cudaStream_t stream) {
  if (s_kv < 0 || s_kv > INT32_MAX) return SMLA_ERR_BAD_SHAPE;
  // with an empty KV every slot is invalid and kv is never read: it may then be NULL
  const void* kv_base = s_kv > 0 ? kv : q;
  smla_status st = check_common(q, kv_base, indices, out, lse, max_logits, s_q, h_q, d_qk, d_v,
                                topk, sm_scale);
  if (st != SMLA_OK || s_q == 0) return st;
  if (attn_sink && !aligned4(attn_sink)) return SMLA_ERR_MISALIGNED;
  if (topk_length && !aligned4(topk_length)) return SMLA_ERR_MISALIGNED;
  CUtensorMap qm, kvm;
  if (!make_map(&qm, q, static_cast<uint64_t>(s_q) * h_q, d_qk, 64)) return SMLA_ERR_TENSOR_MAP;
  // an empty KV still needs a one-row map; every slot is then invalid and never read
  if (!make_map(&kvm, kv_base, s_kv > 0 ? static_cast<uint64_t>(s_kv) : 1u, d_qk, 1))
    return SMLA_ERR_TENSOR_MAP;
  FwdParams p{};
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
  p.s_q_per_req = 1;
  p.page_block = 1;
  p.max_blocks = 1;
  p.pool_rows = s_kv;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  return dispatch<false>(d_qk, topk_length != nullptr, qm, kvm, p, stream);
}

smla_status sparse_mla_fwd_paged(const void* q, const void* kv_pool, int64_t pool_rows,
                                 const int32_t* block_table, int max_blocks, int page_block,
                                 const int32_t* seqlens_k, int64_t s_kv_per_req, int s_q_per_req,
                                 const int32_t* indices, const int32_t* topk_length,
                                 const float* attn_sink, float sm_scale, int d_v, void* out,
                                 float* lse, float* max_logits, int64_t s_q, int h_q, int d_qk,
                                 int topk, cudaStream_t stream) {
  smla_status st = check_common(q, kv_pool, indices, out, lse, max_logits, s_q, h_q, d_qk, d_v,
                                topk, sm_scale);
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
  FwdParams p{};
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
  p.block_table = block_table;
  p.seqlens_k = seqlens_k;
  p.max_blocks = max_blocks;
  p.page_block = page_block;
  p.s_q_per_req = s_q_per_req;
  p.pool_rows = pool_rows;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  return dispatch<true>(d_qk, topk_length != nullptr, qm, kvm, p, stream);
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
  }
  return "unknown status";
}

int sparse_mla_abi_version(void) { return SMLA_ABI_VERSION; }

}  // extern "C"
