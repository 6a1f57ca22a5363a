// Sparse MLA attention backward (DSA top-k) for sm_103a.  Included by sparse_mla_fwd.cu inside
// namespace smla::(anonymous): it shares that file's bounded waits, status word, tensor-map
// encoding and argument checks.
//
// The operation (FlashMLA PR #198, "Summary" item 1: the sparse MLA backward for the absorbed
// shape, dK / dV scattered into the shared latent rows with fp32 atomics): the gradients of
// L = sum dO * O through the forward of PR #196 / #216 / #198 item 2.  For row t, head h and the
// counted slots s (latent row r_s, key k_s = kv[r_s, :d_qk], value v_s = kv[r_s, :d_v]):
//   p_s  = exp(sm_scale q.k_s - lse_full),   lse_full = ln(exp(lse) + [sink] exp(sink_h))
//   D    = <dO, O>,   dS_s = p_s (<dO, v_s> - D)
//   dq_h += sm_scale dS_s k_s,   dkv[r_s, :d_qk] += sm_scale dS_s q_h,   dkv[r_s, :d_v] += p_s dO_h
//   dsink[h] += -exp(sink_h - lse_full) D
// lse is the forward's (natural log, sink excluded) and O the forward's bf16 output.
//
// Work item = (token, group of 64 heads), one CTA each.  Per 64-key block of the row:
//   [S^T | dP^T] [64 keys x (64 + 64)] = K [Q; dO]^T   (M=64, N=128, K=512; then the rope
//                             columns add K_rope Q_rope^T to S^T alone with N=64; TMEM)
//   P^T, dS'^T = sm_scale P (dP - D)  -> shared memory as bf16 [keys][heads] (SW128)
//   dQ^T [d_qk x 64 heads] += K^T dS'^T           (M=128 (+64 for the rope), N=64, K=64 keys;
//                                                  TMEM, accumulated over the row's blocks)
//   dKV^T [d x 64 keys]     = Q^T dS' + dO^T P    (per 128-row chunk of d, K=64 heads; TMEM),
//                             drained into fp32 reductions on dkv
// A tcgen05.mma costs about the same time for N = 64 as for N = 128, so S and dP, which share
// their B rows (the block's kv rows), run as one N = 128 product with the keys as M: half the
// instructions of two M=64 x N=64 products.  With keys on TMEM lanes, each math thread holds two
// keys and sixteen heads, and the masking of invalid slots is per lane.
// The fp32 reductions are the longest job and set the block period, so they run on eight warps
// of their own (two per TMEM lane quadrant, 32 keys each: more reductions in flight), out of a
// TMEM buffer of their own, fed by an MMA issuer of their own: the next block's gather, S, dP,
// P / dS' and dQ proceed while the previous block drains.  Issuer B starts a block's dKV^T
// chunks once dQ^T of that block has run, so they fill the tensor pipe while the next block is
// gathered instead of competing with S, dP and dQ^T.
// With the reductions off the chain, the gather of the next block (which may start only once
// dQ^T has read the single kv stage) is the longest step left on it; TMA issue throughput grows
// with the number of issuing warps, so ten warps gather.
// Warp roles (768 threads, six warpgroups):
//   warp 0        issuer A: S^T / dP^T, dQ^T (one thread); owns TMEM
//   warps 1-2, 16-23  gather: the block's kv rows with TMA gather4 (warp 1 also loads Q and dO
//                 and publishes the row table)
//   warp 3        issuer B: dKV^T chunks (one thread)
//   warps 4-7     math (TMEM lane quadrants 0-3): D / lse prologue, P and dS', dq epilogue
//   warps 8-15    drain (lane quadrant warp % 4, keys 32 ((warp - 8) / 4) + 0..31): dKV^T
//                 chunks -> fp32 reductions on dkv
// 768 threads launch with 80 registers each; setmaxnreg gives the math warpgroup 120 and the
// others 72, which uses the launch's 61440 registers exactly.
// TMEM: dQ^T chunks at columns 0, 64, 128, 192 (+256 for the rope rows); S at 320, dP at 384
// and the dKV^T buffer at 448.  One dKV^T buffer is enough: the drain warps hand it back as soon
// as a chunk is in their registers, long before its reductions end, and the columns it frees let
// S and dP have buffers of their own, so dP does not wait for S to be read.

constexpr int kBwdThreads = 768;
constexpr int kBwdMathWarp0 = 4;
constexpr int kBwdDrainWarp0 = 8;
constexpr int kBwdIssuerB = 3;
constexpr int kBwdGatherWarps = 10;                // warps 1, 2, 16-23
constexpr int kBwdRowSlots = 4;                    // blocks whose row table may be live at once
constexpr int kBwdMathRegs = 120;                  // 128 x 120 + 640 x 72 = 61440 = 768 x 80
constexpr int kBwdOtherRegs = 72;
constexpr uint32_t kBwdTmemS = 320, kBwdTmemDP = 384, kBwdTmemX = 448;

struct BwdParams {
  const int32_t* indices;      // [s_q, topk]
  const int32_t* topk_length;  // [s_q] or null
  const float* attn_sink;      // [h_q] or null
  const float* lse;            // [s_q, h_q], natural log, sink excluded
  const __nv_bfloat16* out;    // [s_q, h_q, 512]
  const __nv_bfloat16* dout;   // [s_q, h_q, 512]
  float* dq;                   // [s_q, h_q, d_qk]
  float* dkv;                  // [s_kv, d_qk], accumulated
  float* dsink;                // [h_q] or null, accumulated
  float sm_scale;
  int64_t s_q;
  int64_t s_kv;
  int h_q;
  int topk;
  int n_groups;
  uint64_t wait_limit_ns;
};

// tcgen05.ld 16x32bx2, 16 columns per half, halves 16 columns apart: threads 0-15 read lanes
// base + t at columns col .. col+15, threads 16-31 read lanes base + t - 16 at col+16 .. col+31
__device__ __forceinline__ void tmem_ld_16x32bx2_x16_off16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// TMA row coordinate of slot j of row t (j < L): the kv row, or -1 when the slot does not count
__device__ __forceinline__ int bwd_row(const BwdParams& p, const int32_t* idx_row, int j, int L) {
  if (j >= L) return -1;
  const int v = __ldg(idx_row + j);
  return (v >= 0 && static_cast<int64_t>(v) < p.s_kv) ? v : -1;
}

template <int D_QK>
__global__ void __launch_bounds__(kBwdThreads, 1)
    sparse_mla_bwd_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap do_map,
                          const __grid_constant__ CUtensorMap kv_map, const BwdParams p) {
  constexpr int kChunks = D_QK / 64;                 // 64-column chunks of q / kv rows
  constexpr int kQkSteps = D_QK / 16;
  constexpr int kDkvChunks = (D_QK + 127) / 128;     // 128-row chunks of d (the last may be 64)
  constexpr bool kRope = (D_QK % 128) != 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // column chunk c (64 columns) of Q and of dO side by side: Q rows at sQD + 16 KB c, dO rows
  // 8 KB further (the rope chunk c = 8 holds Q rows only), so that the 128 rows [Q; dO] of a
  // chunk form one K-major operand
  uint8_t* sQD = smem;
  uint8_t* sKV = sQD + kChunks * 8192 + 8 * 8192;     // [64 keys][D_QK], kChunks x 8 KB
  uint8_t* sP = sKV + kChunks * 8192;                 // [64 keys][64 heads] bf16
  uint8_t* sDS = sP + 8192;                           // [64 keys][64 heads] bf16 (sm_scale dS)

  __shared__ __align__(8) uint64_t bar_qdo_full, bar_kv_full, bar_kv_empty, bar_s_full,
      bar_p_full, bar_tiles_free, bar_dq_full, bar_final_a, bar_final_b;
  __shared__ __align__(8) uint64_t bar_x_full, bar_x_free, bar_rows_full[kBwdRowSlots];
  __shared__ int32_t s_rows[kBwdRowSlots][64];
  __shared__ float s_delta[64];
  __shared__ float s_lse2[64];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort = &abort_flag;
  const uint64_t lim = p.wait_limit_ns;
  const int64_t item = blockIdx.x;
  const int64_t t = item / p.n_groups;
  const int g = static_cast<int>(item % p.n_groups);
  const int32_t* idx_row = p.indices + t * static_cast<int64_t>(p.topk);
  const int L = p.topk_length ? min(max(__ldg(p.topk_length + t), 0), p.topk) : p.topk;
  const int nb = (L + 63) / 64;                       // blocks of this row (uniform for all roles)

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar_qdo_full), 1);
    mbar_init(smem_u32(&bar_kv_full), 1);
    mbar_init(smem_u32(&bar_kv_empty), 1);
    mbar_init(smem_u32(&bar_s_full), 1);
    mbar_init(smem_u32(&bar_p_full), 128);
    mbar_init(smem_u32(&bar_tiles_free), 2);          // dQ^T (issuer A) and dKV^T (issuer B)
    mbar_init(smem_u32(&bar_dq_full), 1);
    mbar_init(smem_u32(&bar_final_a), 1);
    mbar_init(smem_u32(&bar_final_b), 1);
    mbar_init(smem_u32(&bar_x_full), 1);
    mbar_init(smem_u32(&bar_x_free), 8);
    for (int i = 0; i < kBwdRowSlots; ++i) mbar_init(smem_u32(&bar_rows_full[i]), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int64_t qrow = t * p.h_q + static_cast<int64_t>(g) * 64;   // first (token, head) row

  if (warp >= kBwdMathWarp0 && warp < kBwdMathWarp0 + 4) {
    reg_alloc<kBwdMathRegs>();
    // ======================================================== math (see below)
    // P / dS' per block and the dq epilogue of the item
    const int q = warp - kBwdMathWarp0;
    const int mt = tid - kBwdMathWarp0 * 32;         // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // per-item prologue: D = <dO, O> and lse_full * log2(e) for each of the 64 heads (two
    // threads per head, 256 columns each), and the sink's gradient
    {
      const int h = mt >> 1, half = mt & 1;
      const int64_t r = (qrow + h) * 512 + half * 256;
      const uint4* a = reinterpret_cast<const uint4*>(p.dout + r);
      const uint4* o = reinterpret_cast<const uint4*>(p.out + r);
      float acc = 0.f;
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const uint4 x = __ldg(a + k), y = __ldg(o + k);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
          const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
          acc = fmaf(fx.x, fy.x, acc);
          acc = fmaf(fx.y, fy.y, acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      if (half == 0) {
        const int head = g * 64 + h;
        const float lse = __ldg(p.lse + t * p.h_q + head);
        float lf = lse;
        if (p.attn_sink) {
          const float sk = __ldg(p.attn_sink + head);
          const float hi = fmaxf(lse, sk);
          lf = (hi == INFINITY) ? INFINITY : hi + log1pf(expf(fminf(lse, sk) - hi));
          if (p.dsink) atomicAdd(p.dsink + head, -expf(sk - lf) * acc);
        }
        s_delta[h] = acc;
        s_lse2[h] = lf * kLog2e;
      }
    }
    named_bar_sync(1, 128);
    // 16x256b fragments of S^T and dP^T (M=64 layout: keys 16q..16q+15 in lanes 0-15 of
    // quadrant q): this thread holds keys kA = 16q + lane/4 and kB = kA + 8, and heads
    // 8i + 2(lane&3) + {0,1}, whose D and lse it keeps in registers
    const int kA = 16 * q + (lane >> 2), kB = kA + 8;
    const int cpair = 2 * (lane & 3);
    const float c2 = p.sm_scale * kLog2e;
    float dh[16], lh[16];
#pragma unroll
    for (int i8 = 0; i8 < 8; ++i8)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        dh[2 * i8 + e] = s_delta[8 * i8 + cpair + e];
        lh[2 * i8 + e] = s_lse2[8 * i8 + cpair + e];
      }
    for (int b = 0; b < nb && !*abort; ++b) {
      const int rs = b % kBwdRowSlots;
      wait_or_flag(smem_u32(&bar_kv_full), b & 1, abort, lim);   // also publishes s_rows[rs]
      wait_or_flag(smem_u32(&bar_s_full), b & 1, abort, lim);
      SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, b, kTrSReady);
      tc_fence_after();
      float sv[32], dv[32];
#pragma unroll
      for (int i8 = 0; i8 < 8; ++i8) {
        uint32_t r4[4];
        tmem_ld_16x256b(tmem + lane_base + kBwdTmemS + 8 * i8, r4);
#pragma unroll
        for (int e = 0; e < 4; ++e) sv[4 * i8 + e] = __uint_as_float(r4[e]);
      }
#pragma unroll
      for (int i8 = 0; i8 < 8; ++i8) {
        uint32_t d4[4];
        tmem_ld_16x256b(tmem + lane_base + kBwdTmemDP + 8 * i8, d4);
#pragma unroll
        for (int e = 0; e < 4; ++e) dv[4 * i8 + e] = __uint_as_float(d4[e]);
      }
      const bool okA = s_rows[rs][kA] >= 0, okB = s_rows[rs][kB] >= 0;
      tmem_ld_wait();
      // P^T and dS'^T as packed bf16 pairs: [i8][0] P key kA, [1] P key kB, [2] dS' kA, [3] dS' kB.
      // They are formed before the wait for the tiles, which is a wait for dKV^T(b-1) and so for
      // the drains of block b-1.
      uint32_t pk[8][4];
#pragma unroll
      for (int i8 = 0; i8 < 8; ++i8) {
        float pa[2], pb[2], da[2], db[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pa[e] = okA ? fast_exp2(fmaf(sv[4 * i8 + e], c2, -lh[2 * i8 + e])) : 0.f;
          pb[e] = okB ? fast_exp2(fmaf(sv[4 * i8 + 2 + e], c2, -lh[2 * i8 + e])) : 0.f;
          da[e] = p.sm_scale * pa[e] * (dv[4 * i8 + e] - dh[2 * i8 + e]);
          db[e] = p.sm_scale * pb[e] * (dv[4 * i8 + 2 + e] - dh[2 * i8 + e]);
        }
        pk[i8][0] = pack_bf16x2(pa[0], pa[1]);
        pk[i8][1] = pack_bf16x2(pb[0], pb[1]);
        pk[i8][2] = pack_bf16x2(da[0], da[1]);
        pk[i8][3] = pack_bf16x2(db[0], db[1]);
      }
      // the previous block's P / dS' tiles have been read by every MMA (dQ^T and dKV^T)
      if (b >= 1) wait_or_flag(smem_u32(&bar_tiles_free), (b - 1) & 1, abort, lim);
      const int swA = kA & 7, swB = kB & 7;
      const int off = 2 * cpair;
#pragma unroll
      for (int i8 = 0; i8 < 8; ++i8) {
        *reinterpret_cast<uint32_t*>(sP + kA * 128 + ((i8 ^ swA) << 4) + off) = pk[i8][0];
        *reinterpret_cast<uint32_t*>(sP + kB * 128 + ((i8 ^ swB) << 4) + off) = pk[i8][1];
        *reinterpret_cast<uint32_t*>(sDS + kA * 128 + ((i8 ^ swA) << 4) + off) = pk[i8][2];
        *reinterpret_cast<uint32_t*>(sDS + kB * 128 + ((i8 ^ swB) << 4) + off) = pk[i8][3];
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bar_p_full));            // also: S and dP have been read
      SMLA_TRACE_EVENT_IF(q == 0 && lane == 0, b, kTrPReady);
    }
    // ---- dq of this item: dQ^T chunk c holds rows d, columns = heads
    float* dq = p.dq + qrow * D_QK;
    if (nb > 0) {
      wait_or_flag(smem_u32(&bar_dq_full), 0, abort, lim);
      tc_fence_after();
    }
#pragma unroll 1
    for (int c = 0; c < kDkvChunks; ++c) {
      const bool rope = kRope && c == 4;
      const int d = rope ? 512 + 16 * q + lane : 128 * c + 32 * q + lane;
#pragma unroll 1
      for (int h16 = 0; h16 < 4; ++h16) {
        uint32_t r[16];
        if (nb > 0) {
          tmem_ld16(tmem + lane_base + 64 * c + 16 * h16, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = 0u;
        }
        if (!rope || lane < 16) {
#pragma unroll
          for (int j = 0; j < 16; ++j) dq[static_cast<int64_t>(16 * h16 + j) * D_QK + d] = __uint_as_float(r[j]);
        }
      }
    }
  } else {
    reg_dealloc<kBwdOtherRegs>();
    if (warp == 0) {
      // ======================================================== issuer A: S, dP, dQ^T
      if (lane == 0 && nb > 0) {
        constexpr uint32_t id_sd = make_idesc_bf16(64, 128, false, false);  // [S^T | dP^T]
        constexpr uint32_t id_s = make_idesc_bf16(64, 64, false, false);    // S^T, rope columns
        constexpr uint32_t id_dq = make_idesc_bf16(128, 64, true, true);
        constexpr uint32_t id_dq64 = make_idesc_bf16(64, 64, true, true);
        const uint64_t qd_k = make_sdesc_sw128(smem_u32(sQD), 16, 1024);    // [Q; dO] rows, K-major
        const uint64_t kv_k = make_sdesc_sw128(smem_u32(sKV), 16, 1024);    // K / V rows, K-major
        const uint64_t kv_mn = make_sdesc_sw128(smem_u32(sKV), 8192, 1024); // K^T, MN-major
        const uint64_t ds_mn = make_sdesc_sw128(smem_u32(sDS), 8192, 1024); // dS'^T operand, MN-major
        wait_or_flag(smem_u32(&bar_qdo_full), 0, abort, lim);
        for (int b = 0; b < nb && !*abort; ++b) {
          wait_or_flag(smem_u32(&bar_kv_full), b & 1, abort, lim);
          SMLA_TRACE_EVENT(b, kTrGatherIssue);
          tc_fence_after();
          // S and dP: their columns were read by the math warps before p_full(b-1), which this
          // thread waited for before dQ^T(b-1)
          // [S^T | dP^T] (keys x (64 heads of S, 64 of dP)) = K [Q; dO]^T over the 512 value
          // columns in one N = 128 chain, then the rope columns add to S^T alone
#pragma unroll 4
          for (int ks = 0; ks < 32; ++ks)
            umma_ss(tmem + kBwdTmemS, kv_k + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4),
                    qd_k + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), id_sd, ks > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 32; ks < kQkSteps; ++ks)
            umma_ss(tmem + kBwdTmemS, kv_k + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4),
                    qd_k + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), id_s, 1u);
          umma_commit(smem_u32(&bar_s_full));              // S^T and dP^T
          SMLA_TRACE_EVENT(b, kTrQkIssue);
          wait_or_flag(smem_u32(&bar_p_full), b & 1, abort, lim);
          tc_fence_after();
          // dQ^T += K^T dS'^T over this block's 64 keys
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_ss(tmem + 64 * c, kv_mn + ((2 * c * 8192 + ks * 2048) >> 4), ds_mn + ((ks * 2048) >> 4), id_dq,
                      (b > 0 || ks > 0) ? 1u : 0u);
          if constexpr (kRope) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_ss(tmem + 256, kv_mn + ((8 * 8192 + ks * 2048) >> 4), ds_mn + ((ks * 2048) >> 4), id_dq64,
                      (b > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar_kv_empty));          // S, dP and dQ^T have read the stage
          umma_commit(smem_u32(&bar_tiles_free));        // ... and dQ^T the dS' tile
          SMLA_TRACE_EVENT(b, kTrPvIssue);
        }
        umma_commit(smem_u32(&bar_dq_full));
        umma_commit(smem_u32(&bar_final_a));
        wait_drain(smem_u32(&bar_final_a), 0, lim);
      }
      __syncwarp();
    } else if (warp == kBwdIssuerB) {
      // ======================================================== issuer B: dKV^T chunks
      if (lane == 0 && nb > 0) {
        constexpr uint32_t id_kv = make_idesc_bf16(128, 64, true, false);
        constexpr uint32_t id_kv64 = make_idesc_bf16(64, 64, true, false);
        const uint64_t q_mn = make_sdesc_sw128(smem_u32(sQD), 16384, 1024);        // Q^T, MN-major
        const uint64_t do_mn = make_sdesc_sw128(smem_u32(sQD) + 8192, 16384, 1024); // dO^T, MN-major
        const uint64_t ds_k = make_sdesc_sw128(smem_u32(sDS), 16, 1024);    // dS' operand, K-major
        const uint64_t p_k = make_sdesc_sw128(smem_u32(sP), 16, 1024);      // P operand, K-major
        uint32_t xu = 0;                              // fills of the dKV^T buffer so far
        wait_or_flag(smem_u32(&bar_qdo_full), 0, abort, lim);
        for (int b = 0; b < nb && !*abort; ++b) {
          // after dQ^T(b) (issuer A's critical chain) has run: dKV^T(b) then fills the tensor
          // pipe while block b+1 is gathered
          wait_or_flag(smem_u32(&bar_kv_empty), b & 1, abort, lim);
#pragma unroll
          for (int c = 0; c < kDkvChunks; ++c) {
            if (xu > 0) wait_or_flag(smem_u32(&bar_x_free), (xu - 1) & 1, abort, lim);
            tc_fence_after();
            const uint32_t col = tmem + kBwdTmemX;
            if (!kRope || c < 4) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_ss(col, q_mn + ((2 * c * 16384 + ks * 2048) >> 4), ds_k + ((ks * 32) >> 4), id_kv,
                        ks > 0 ? 1u : 0u);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_ss(col, do_mn + ((2 * c * 16384 + ks * 2048) >> 4), p_k + ((ks * 32) >> 4), id_kv, 1u);
            } else {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                umma_ss(col, q_mn + ((8 * 16384 + ks * 2048) >> 4), ds_k + ((ks * 32) >> 4), id_kv64,
                        ks > 0 ? 1u : 0u);
            }
            umma_commit(smem_u32(&bar_x_full));
            ++xu;
          }
          umma_commit(smem_u32(&bar_tiles_free));        // P and dS' tiles may be rewritten
          SMLA_TRACE_EVENT(b, kTrEpilogue);
        }
        umma_commit(smem_u32(&bar_final_b));
        wait_drain(smem_u32(&bar_final_b), 0, lim);
      }
      __syncwarp();
    } else if (warp >= kBwdDrainWarp0 && warp < kBwdDrainWarp0 + 8) {
      // ======================================================== drain (see below)
      // dKV^T chunks of every block, in issue order, into fp32 reductions on the selected rows.
      // Warps 8+q and 12+q own TMEM lanes 32q..32q+31 (d = 128c + 32q + lane, or 512 + 16q + lane
      // on lanes 0-15 for the 64 rope rows) and key columns 0-31 and 32-63 of each chunk; the 32
      // lanes of a warp cover 128 contiguous bytes of one kv row.  The reductions are bound by
      // their instruction count, so every one of them carries 32 values: on the rope chunk the
      // two thread halves take different keys.
      const int q = warp & 3, hf = (warp - kBwdDrainWarp0) >> 2;   // lane quadrant, key half
      const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
      uint32_t xu = 0;
      for (int b = 0; b < nb && !*abort; ++b) {
        const int rs = b % kBwdRowSlots;
        // the block's row table (written by the first gather warp before its gathers)
        wait_or_flag(smem_u32(&bar_rows_full[rs]), (b / kBwdRowSlots) & 1, abort, lim);
#pragma unroll
        for (int c = 0; c < kDkvChunks; ++c) {
          wait_or_flag(smem_u32(&bar_x_full), xu & 1, abort, lim);
          SMLA_TRACE_EVENT_IF(c == 0 && q == 0 && hf == 0 && lane == 0, b, kTrSLoaded);
          ++xu;
          tc_fence_after();
          const uint32_t col = kBwdTmemX;
          if (kRope && c == 4) {
            // the 64 rope rows sit on lanes 0-15 of each quadrant: both thread halves take part,
            // threads 16-31 on the second 16 of this warp's 32 keys, so 16 reductions cover them
            uint32_t v[16];
            tmem_ld_16x32bx2_x16_off16(tmem + lane_base + col + 32 * hf, v);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_x_free));
            float* base = p.dkv + 512 + 16 * q + (lane & 15);
            const int k0 = 32 * hf + 16 * (lane >> 4);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int row = s_rows[rs][k0 + k];
              if (row >= 0) atomicAdd(base + static_cast<int64_t>(row) * D_QK, __uint_as_float(v[k]));
            }
          } else {
            float* base = p.dkv + 128 * c + 32 * q + lane;
            // this warp's 32 keys; the buffer goes back once every drain warp has its half
            uint32_t v[32];
            tmem_ld16(tmem + lane_base + col + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            tmem_ld16(tmem + lane_base + col + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_x_free));
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int row = s_rows[rs][32 * hf + k];
              if (row >= 0) atomicAdd(base + static_cast<int64_t>(row) * D_QK, __uint_as_float(v[k]));
            }
          }
        }
      }
      SMLA_TRACE_EVENT_IF(q == 0 && hf == 0 && lane == 0, nb, kTrSent);
    } else {
      // ======================================================== gather (see below)
      // warps 1-2 and 16-23; the first loads the item's Q and dO tiles and publishes each block's
      // row table (TMA row coordinates, -1 for slots that do not count)
      const int gw = warp < 3 ? warp - 1 : warp - 14;   // 0..9
      const bool leader = (gw == 0 && lane == 0);
      if (leader && nb > 0) {
        mbar_arrive_expect_tx(smem_u32(&bar_qdo_full), (kChunks + 8) * 8192u);
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(smem_u32(sQD + c * 16384), &q_map, 64 * c, static_cast<int>(qrow), smem_u32(&bar_qdo_full));
        for (int c = 0; c < 8; ++c)
          tma_load_2d(smem_u32(sQD + c * 16384 + 8192), &do_map, 64 * c, static_cast<int>(qrow), smem_u32(&bar_qdo_full));
      }
      // (4-row group, chunk) items of a block: item gw + 2 (lane + 32 j) for j < kGI
      constexpr int kGI = (16 * kChunks + 32 * kBwdGatherWarps - 1) / (32 * kBwdGatherWarps);
      auto item_of = [&](int j) { return gw + kBwdGatherWarps * (lane + 32 * j); };
      // the rows of block b+1 are loaded while block b is in flight (indices come from HBM)
      auto rows4 = [&](int b, int j) {
        const int r0 = 64 * b + 4 * (item_of(j) & 15);
        return make_int4(bwd_row(p, idx_row, r0, L), bwd_row(p, idx_row, r0 + 1, L), bwd_row(p, idx_row, r0 + 2, L),
                         bwd_row(p, idx_row, r0 + 3, L));
      };
      auto rows2 = [&](int b) {
        return make_int2(bwd_row(p, idx_row, 64 * b + lane, L), bwd_row(p, idx_row, 64 * b + lane + 32, L));
      };
      int4 nxt4[kGI];
      int2 nxt2 = make_int2(-1, -1);
#pragma unroll
      for (int j = 0; j < kGI; ++j) nxt4[j] = make_int4(-1, -1, -1, -1);
      if (nb > 0) {
#pragma unroll
        for (int j = 0; j < kGI; ++j)
          if (item_of(j) < 16 * kChunks) nxt4[j] = rows4(0, j);
        if (gw == 0) nxt2 = rows2(0);
      }
      for (int b = 0; b < nb && !*abort; ++b) {
        int4 cur4[kGI];
#pragma unroll
        for (int j = 0; j < kGI; ++j) cur4[j] = nxt4[j];
        const int2 cur2 = nxt2;
        if (b + 1 < nb) {
#pragma unroll
          for (int j = 0; j < kGI; ++j)
            if (item_of(j) < 16 * kChunks) nxt4[j] = rows4(b + 1, j);
          if (gw == 0) nxt2 = rows2(b + 1);
        }
        if (b >= 1) wait_or_flag(smem_u32(&bar_kv_empty), (b - 1) & 1, abort, lim);
        SMLA_TRACE_EVENT_IF(leader, b, kTrRing);
        if (gw == 0) {
          // slot b % 4 was last read by the drains of block b-4: each drain warp ends them before
          // it takes block b-3's first chunk, so the dKV^T buffer could not take block b-3's
          // second chunk, nor dKV^T(b-2) run, nor the P / dS' tiles of block b-1 be written (the
          // kv_empty(b-1) wait above follows those) before they were done
          const int rs = b % kBwdRowSlots;
          s_rows[rs][lane] = cur2.x;
          s_rows[rs][lane + 32] = cur2.y;
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bar_rows_full[rs]));
            mbar_arrive_expect_tx(smem_u32(&bar_kv_full), kChunks * 8192u);
          }
        }
#pragma unroll
        for (int j = 0; j < kGI; ++j) {
          const int it = item_of(j), chunk = it >> 4;
          if (it < 16 * kChunks)
            tma_gather4(smem_u32(sKV + chunk * 8192 + (it & 15) * 512), &kv_map, 64 * chunk, cur4[j].x, cur4[j].y,
                        cur4[j].z, cur4[j].w, smem_u32(&bar_kv_full));
        }
      }
      // the Q / dO tiles and the last block have landed before this CTA may exit
      if (leader && nb > 0) {
        wait_drain(smem_u32(&bar_qdo_full), 0, lim);
        wait_drain(smem_u32(&bar_kv_full), (nb - 1) & 1, lim);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D_QK>
constexpr size_t bwd_smem_bytes() {
  return (2 * (D_QK / 64) + 10) * 8192 + 1024;
}

// Sets the kernel's shared-memory attribute (before anything is enqueued).
template <int D_QK>
smla_status prepare_bwd() {
  return cudaFuncSetAttribute(sparse_mla_bwd_kernel<D_QK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bwd_smem_bytes<D_QK>())) == cudaSuccess
             ? SMLA_OK
             : SMLA_ERR_LAUNCH;
}

template <int D_QK>
smla_status launch_bwd(const CUtensorMap& qm, const CUtensorMap& dom, const CUtensorMap& kvm, const BwdParams& p,
                       int64_t n_items, cudaStream_t stream) {
  sparse_mla_bwd_kernel<D_QK><<<static_cast<unsigned>(n_items), kBwdThreads, bwd_smem_bytes<D_QK>(), stream>>>(
      qm, dom, kvm, p);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_LAUNCH;
}

smla_status bwd_flat(const void* q, const void* kv, const void* out, const void* dout, const int32_t* indices,
                     const int32_t* topk_length, const float* attn_sink, const float* lse, float sm_scale,
                     int d_v, float* dq, float* dkv, float* dsink, int64_t s_q, int64_t s_kv, int h_q, int d_qk,
                     int topk, cudaStream_t stream) {
  // every argument is checked before anything is enqueued
  if (s_kv < 0) return SMLA_ERR_BAD_SHAPE;
  smla_status st = check_common(q, s_kv > 0 ? kv : q, indices, dq, lse, dq, s_q, h_q, d_qk, d_v, topk, sm_scale);
  if (st != SMLA_OK) return st;
  if (s_q > 0) {
    if (!out || !dout) return SMLA_ERR_NULL_PTR;
    if (!aligned16(out) || !aligned16(dout)) return SMLA_ERR_MISALIGNED;
    if (attn_sink && !aligned4(attn_sink)) return SMLA_ERR_MISALIGNED;
    if (topk_length && !aligned4(topk_length)) return SMLA_ERR_MISALIGNED;
  }
  if (s_kv > 0 && !dkv) return SMLA_ERR_NULL_PTR;
  if ((dkv && !aligned4(dkv)) || (dsink && !aligned4(dsink))) return SMLA_ERR_MISALIGNED;
  // tensor maps and the kernel attribute come before the memsets, so that every error but a
  // failed launch itself is returned before anything is enqueued
  CUtensorMap qm, dom, kvm;
  if (s_q > 0) {
    const uint64_t rows = static_cast<uint64_t>(s_q) * h_q;
    if (!make_map(&qm, q, rows, d_qk, 64) || !make_map(&dom, dout, rows, d_v, 64)) return SMLA_ERR_TENSOR_MAP;
    if (!make_map(&kvm, s_kv > 0 ? kv : q, s_kv > 0 ? static_cast<uint64_t>(s_kv) : 1u, d_qk, 1))
      return SMLA_ERR_TENSOR_MAP;
    st = d_qk == 512 ? prepare_bwd<512>() : prepare_bwd<576>();
    if (st != SMLA_OK) return st;
  }
  // dkv and dsink are accumulated into: they start at zero
  if (s_kv > 0 && cudaMemsetAsync(dkv, 0, static_cast<size_t>(s_kv) * d_qk * sizeof(float), stream) != cudaSuccess)
    return SMLA_ERR_LAUNCH;
  if (dsink && cudaMemsetAsync(dsink, 0, static_cast<size_t>(h_q) * sizeof(float), stream) != cudaSuccess)
    return SMLA_ERR_LAUNCH;
  if (s_q == 0) return SMLA_OK;
  BwdParams p{};
  p.indices = indices;
  p.topk_length = topk_length;
  p.attn_sink = attn_sink;
  p.lse = lse;
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dq = dq;
  p.dkv = dkv;
  p.dsink = attn_sink ? dsink : nullptr;
  p.sm_scale = sm_scale;
  p.s_q = s_q;
  p.s_kv = s_kv;
  p.h_q = h_q;
  p.topk = topk;
  p.n_groups = h_q / kGroupHeads;
  p.wait_limit_ns = kDefaultWaitLimitNs;
  const int64_t n_items = s_q * p.n_groups;
  return d_qk == 512 ? launch_bwd<512>(qm, dom, kvm, p, n_items, stream)
                     : launch_bwd<576>(qm, dom, kvm, p, n_items, stream);
}
