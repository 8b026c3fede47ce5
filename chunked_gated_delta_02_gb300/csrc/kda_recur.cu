// K2: head-parallel chunk recurrence of the KDA chunked forward, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, head, 64-wide slice of V). The CTA walks the chunks
// of its sequence in order and carries its K x 64 slice of the state S (the
// FlashKDA "K2" stage, FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의
// 분리"; the cuLA "chunk gated delta h" + "chunk fwd o" stages, cuLA launch
// blog, section "Status & Roadmap"). Per chunk, with M = [-Tb ; P Tb] from
// the prep kernel and the in-chunk decays measured from the chunk start:
//
//   D1 = M (khat Gamma)          = [-w ; P w]        (128 x K,  UMMA 128xKx64)
//   D2 = M v                     = [-u ; P u]        (128 x 64, UMMA 128x64x64)
//   WQ = [w ; q~ - P w],  q~ = qhat Gamma            (fp16 operand)
//   D2 += WQ S                   = [-U ; O]          (UMMA 128x64xK)
//   U -> fp16, o = scale O -> bf16
//   D3 = k~^T U,  k~ = khat Gamma_last / Gamma       (UMMA 128x64x64)
//   S  = Gamma_last S + D3                           (fp32 master in registers)
//
// Gamma_i is the product of the per-token decays alpha up to token i (all
// factors <= 1, formed as products, never as quotients). U holds the
// delta-rule residuals v - prediction of the chunk; O the inter-chunk term
// q~ S plus the intra-chunk term P U.
//
// The prep kernel hands over M, khat Gamma and k~ (as swizzled operand images),
// q~ and Gamma_last per chunk; v comes straight from the input by TMA.
//
// Warp roles (the S-independent work of chunk n+1 overlaps the state chain of
// chunk n):
//   chain group, warps 0-3: D2 += WQ S, U and o, D3 = k~^T U, S update.
//   prep group, warps 4-11: stages the chunk's operands (bulk copies and one
//     TMA tile of v), converts v to fp16, issues D1 and D2, and forms WQ.
// The groups hand over through mbarriers. Every wait gives up after a bounded
// time; the groups then agree (barrier with OR-reduction) to stop, drain their
// tensor-core work, free TMEM and report KDA_DEVICE_WAIT_TIMEOUT.
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kChainThreads = 128;
constexpr int kPrepGroupThreads = 256;
constexpr int kRecThreads = kChainThreads + kPrepGroupThreads;
constexpr int kBV = 64;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clocks per wait
constexpr int kBarPrep = 1, kBarChain = 2;        // named barrier ids (0 is __syncthreads)

template <int K>
struct RecLayout {
  // byte offsets from the 1024-aligned dynamic shared memory base
  static constexpr uint32_t kPanel64 = 64 * 128;                 // 64 rows x 128 B
  static constexpr uint32_t Mh = 0;                              // 128 x 64  K-major (A of D1, D2)
  static constexpr uint32_t kG = Mh + 128 * 128;                 // 64 x K    MN-major (B of D1)
  static constexpr uint32_t vh = kG + (K / 64) * kPanel64;       // 64 x 64   MN-major (B of D2)
  static constexpr uint32_t WQ = vh + kPanel64;                  // 128 x K   K-major (A of MMA1)
  static constexpr uint32_t Sh = WQ + (K / 64) * 128 * 128;      // K x 64    MN-major (B of MMA1)
  static constexpr uint32_t kT = Sh + K * 128;                   // 2 x (64 x 128 MN-major) (A of MMA2)
  static constexpr uint32_t Uh = kT + 2 * 2 * kPanel64;          // 64 x 64   MN-major (B of MMA2)
  static constexpr uint32_t qt = Uh + kPanel64;                  // 64 x K    q~ image (64-channel panels)
  static constexpr uint32_t rv = qt + 64 * K * 2;                // bf16 v [64][64]
  static constexpr uint32_t misc = rv + 64 * kBV * 2;
  static constexpr uint32_t bytes = misc + 4096 + 1024;          // + misc + alignment slack
};

// Small per-CTA state after the operand buffers.
template <int K>
struct RecMisc {
  uint64_t bar_d12, bar_wq_full, bar_mma1, bar_mma2, bar_exit, bar_in, bar_q;
  uint32_t tmem_slot;
  int err;
  float gam[2][K];           // per chunk (double-buffered): product of alpha over the chunk
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

template <int K>
__global__ void __launch_bounds__(kRecThreads, 1)
recur_tc_kernel(const Problem p, const __grid_constant__ TmaMaps maps) {
  using Lay = RecLayout<K>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  __nv_bfloat16 *rv = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rv);
  RecMisc<K> &ms = *reinterpret_cast<RecMisc<K> *>(sm + Lay::misc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int VT = p.V / kBV;
  const int bid = blockIdx.x;
  const int r = bid / (p.H * VT);
  const int h = (bid / VT) % p.H;
  const int v0 = (bid % VT) * kBV;
  if (p.flag && *p.flag != kDevOk) return;
  const int s = p.cu ? p.order[r] : r;
  const SeqInfo si = seq_info(p, s);
  const uint32_t sbase = umma::smem_u32(sm);
  const int nch = (si.len + kChunk - 1) / kChunk;
  const bool is_chain = warp < 4;
  const int pt = tid - kChainThreads;   // prep thread index (prep group only)

  // ---- set-up: zero the k~ operands (rows >= K stay zero when K = 64), TMEM, barriers
  for (int x = tid; x < (int)(2 * 2 * Lay::kPanel64 / 16); x += kRecThreads)
    reinterpret_cast<uint4 *>(sm + Lay::kT)[x] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(&ms.bar_d12, 1);
    umma::mbar_init(&ms.bar_wq_full, 1);
    umma::mbar_init(&ms.bar_mma1, 1);
    umma::mbar_init(&ms.bar_mma2, 1);
    umma::mbar_init(&ms.bar_exit, 2);
    umma::mbar_init(&ms.bar_in, 1);
    umma::mbar_init(&ms.bar_q, 1);
    umma::mbar_fence_init();
    ms.err = 0;
  }
  // chain threads: state master S[k][0:64] (fp32, thread k) and its fp16 operand copy
  float S[kBV];
  if (is_chain && tid < K) {
#pragma unroll
    for (int v = 0; v < kBV; ++v)
      S[v] = p.init ? p.init[(((long long)s * p.H + h) * p.V + v0 + v) * K + tid] : 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 w;
      w.x = pack_half2(S[8 * c + 0], S[8 * c + 1]);
      w.y = pack_half2(S[8 * c + 2], S[8 * c + 3]);
      w.z = pack_half2(S[8 * c + 4], S[8 * c + 5]);
      w.w = pack_half2(S[8 * c + 6], S[8 * c + 7]);
      *reinterpret_cast<uint4 *>(sm + Lay::Sh + umma::sw128_chunk(tid, c)) = w;
    }
  }
  // Operands of chunk n, issued by one prep thread, in two groups:
  //   bar_in: M and khat Gamma (bulk copies of the pre-swizzled images) and the v tile
  //           (64 x 64 at column v0, one TMA copy; tokens past T read as zeros, tokens of the
  //           next packed sequence are zeroed after arrival); consumed by D1 / D2.
  //   bar_q:  q~ (image), k~ (image, into buffer n & 1) and Gamma_last (into slot n & 1);
  //           q~ is consumed by the WQ rows, k~ by D3, Gamma_last by the state update.
  auto stage_in = [&](int n) {
    if (pt == 0) {
      const long long slot = ((long long)si.chunk0 + n) * p.H + h;
      umma::mbar_arrive_expect_tx(&ms.bar_in, 2 * kChunk * kChunk * 2 + kChunk * K * 2 + kChunk * kBV * 2);
      umma::bulk_g2s(sm + Lay::Mh, p.mats + slot * (2 * kChunk * kChunk), 2 * kChunk * kChunk * 2, &ms.bar_in);
      umma::bulk_g2s(sm + Lay::kG, p.kgimg + slot * (kChunk * K), kChunk * K * 2, &ms.bar_in);
      umma::tma_load_4d(rv, &maps.v, v0, h, si.t0 + n * kChunk, si.b, &ms.bar_in);
    }
  };
  auto stage_q = [&](int n) {
    if (pt == 0) {
      const long long slot = ((long long)si.chunk0 + n) * p.H + h;
      umma::mbar_arrive_expect_tx(&ms.bar_q, 2 * kChunk * K * 2 + K * 4);
      umma::bulk_g2s(sm + Lay::qt, p.qtb + slot * (kChunk * K), kChunk * K * 2, &ms.bar_q);
      umma::bulk_g2s(sm + Lay::kT + (n & 1) * (2 * Lay::kPanel64), p.ktimg + slot * (kChunk * K), kChunk * K * 2,
                     &ms.bar_q);
      umma::bulk_g2s(&ms.gam[n & 1][0], p.gam + slot * K, K * 4, &ms.bar_q);
    }
  };
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (!is_chain && nch > 0) {
    stage_in(0);
    stage_q(0);
  }
  const uint32_t tmem = ms.tmem_slot;
  const uint32_t tD1 = tmem, tD3 = tmem + 256;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool bad = false;   // this thread saw a wait time out
  uint32_t in_done = 0, q_done = 0;   // completed bar_in / bar_q phases seen by this thread

  auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
    if (bad) return;
    if (!umma::mbar_wait_bounded(bar, parity, kWaitLimit)) {
      atomicExch(&ms.err, 1);
      bad = true;
      return;
    }
    umma::fence_after_sync();
  };

  if (is_chain) {
    // ======================= chain group =======================
    for (int n = 0; n < nch; ++n) {
      if (umma::bar_red_or(kBarChain, kChainThreads, bad || *(volatile int *)&ms.err != 0)) break;
      const uint32_t par = (uint32_t)(n & 1);
      const uint32_t tD2 = tmem + 128 + 64 * (n & 1);
      const int t0 = si.t0 + n * kChunk;
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_wq_full, par);
      const float gam = (tid < K) ? ms.gam[n & 1][tid] : 0.f;   // read before MMA1: the slot is reused
      if (tid == 0 && !bad) {   // D2 += WQ S  ->  [-U ; O]
        const uint32_t id = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks) {
          const uint64_t a = umma::sdesc_sw128(sbase + Lay::WQ + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t b = umma::sdesc_sw128(sbase + Lay::Sh + ks * 2048, K * 128, 1024);
          umma::mma_f16_ss(tD2, a, b, id, 1);
        }
        umma::commit(&ms.bar_mma1);
      }
      wait_bar(&ms.bar_mma1, par);
      // U (rows < 64) -> fp16 operand; o = scale * O (rows >= 64) -> bf16 global
#pragma unroll 1
      for (int c0 = 0; c0 < kBV; c0 += 16) {
        float x[16];
        umma::tmem_ld16(tD2 + lane_base + c0, x);
        umma::tmem_ld_wait();
        if (tid < kChunk) {
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint4 w;
            w.x = pack_half2(-x[8 * hc + 0], -x[8 * hc + 1]);
            w.y = pack_half2(-x[8 * hc + 2], -x[8 * hc + 3]);
            w.z = pack_half2(-x[8 * hc + 4], -x[8 * hc + 5]);
            w.w = pack_half2(-x[8 * hc + 6], -x[8 * hc + 7]);
            *reinterpret_cast<uint4 *>(sm + Lay::Uh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
          }
        } else if (tid - kChunk < L && !bad) {
          __nv_bfloat16 ob[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) ob[j] = __float2bfloat16_rn(p.scale * x[j]);
          uint4 *dst = reinterpret_cast<uint4 *>(p.o + tok_row(p, si.b, t0 + tid - kChunk, h) * p.V + v0 + c0);
          dst[0] = *reinterpret_cast<const uint4 *>(&ob[0]);
          dst[1] = *reinterpret_cast<const uint4 *>(&ob[8]);
        }
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarChain, kChainThreads);
      if (tid == 0 && !bad) {   // D3 = k~^T U
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, kBV, 1, 1);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
          const uint64_t a = umma::sdesc_sw128(sbase + Lay::kT + (n & 1) * (2 * Lay::kPanel64) + ks * 2048,
                                               Lay::kPanel64, 1024);
          const uint64_t b = umma::sdesc_sw128(sbase + Lay::Uh + ks * 2048, Lay::kPanel64, 1024);
          umma::mma_f16_ss(tD3, a, b, id, ks > 0);
        }
        umma::commit(&ms.bar_mma2);
      }
      wait_bar(&ms.bar_mma2, par);
      // S = gamma S + D3 (thread = channel), fp16 copy for the next chunk
      if (tid < K) {
#pragma unroll
        for (int c0 = 0; c0 < kBV; c0 += 16) {
          float x[16];
          umma::tmem_ld16(tD3 + lane_base + c0, x);
          umma::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) S[c0 + j] = fmaf(gam, S[c0 + j], x[j]);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint4 w;
            const float *sv = &S[c0 + 8 * hc];
            w.x = pack_half2(sv[0], sv[1]);
            w.y = pack_half2(sv[2], sv[3]);
            w.z = pack_half2(sv[4], sv[5]);
            w.w = pack_half2(sv[6], sv[7]);
            *reinterpret_cast<uint4 *>(sm + Lay::Sh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
          }
        }
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarChain, kChainThreads);
    }
  } else {
    // ======================= prep group =======================
    for (int n = 0; n < nch; ++n) {
      const uint32_t par = (uint32_t)(n & 1);
      const uint32_t tD2 = tmem + 128 + 64 * (n & 1);
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_in, par);
      in_done += bad ? 0u : 1u;
      if (L < kChunk) {   // v rows past the sequence end (next packed sequence or zero fill): zero them
        for (int x = pt; x < (kChunk - L) * (kBV / 8); x += kPrepGroupThreads) {
          const int i = L + x / (kBV / 8), c8 = x % (kBV / 8);
          *reinterpret_cast<uint4 *>(rv + i * kBV + 8 * c8) = make_uint4(0, 0, 0, 0);
        }
      }
      if (umma::bar_red_or(kBarPrep, kPrepGroupThreads, bad || *(volatile int *)&ms.err != 0)) break;
      if (pt == 0 && !bad) {   // D1 = M (khat Gamma): both operands arrived by copy
        umma::fence_after_sync();
        const uint32_t id1 = umma::idesc_f16(128, K, 0, 1);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tD1, umma::sdesc_sw128(sbase + Lay::Mh + ks * 32, 16, 1024),
                           umma::sdesc_sw128(sbase + Lay::kG + ks * 2048, Lay::kPanel64, 1024), id1, ks > 0);
      }
      // -- v tile -> fp16 operand (2 chunks of 8 values per thread)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int x = pt + kPrepGroupThreads * j;
        const int i = x >> 3, cc = x & 7;
        const uint4 raw = *reinterpret_cast<const uint4 *>(rv + i * kBV + 8 * cc);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
        const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
        *reinterpret_cast<uint4 *>(sm + Lay::vh + umma::sw128_chunk(i, cc)) =
            make_uint4(pack_half2(f0.x, f0.y), pack_half2(f1.x, f1.y), pack_half2(f2.x, f2.y),
                       pack_half2(f3.x, f3.y));
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarPrep, kPrepGroupThreads);   // vh complete; the v tile is consumed
      if (pt == 0 && !bad) {   // D2 = M v; the commit covers D1 too
        umma::fence_after_sync();
        const uint32_t id2 = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tD2, umma::sdesc_sw128(sbase + Lay::Mh + ks * 32, 16, 1024),
                           umma::sdesc_sw128(sbase + Lay::vh + ks * 2048, Lay::kPanel64, 1024), id2, ks > 0);
        umma::commit(&ms.bar_d12);
      }
      wait_bar(&ms.bar_d12, par);
      if (n + 1 < nch) stage_in(n + 1);   // M, khat Gamma and v of chunk n are consumed
      wait_bar(&ms.bar_q, par);
      q_done += bad ? 0u : 1u;

      // -- WQ rows: w = -D1 (rows < 64), Q' = q~ - D1 (rows >= 64); WQ must be free (MMA1 of n-1 done)
      if (n > 0) wait_bar(&ms.bar_mma1, par ^ 1u);
      {
        const int row = (warp & 3) * 32 + lane;        // TMEM lane of this warp's quadrant
        const int cbeg = (warp >= 8) ? K / 2 : 0;       // warps 4-7: low half of the columns
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + K / 2; c0 += 16) {
          float x[16];
          umma::tmem_ld16(tD1 + lane_base + c0, x);
          umma::tmem_ld_wait();
          if (row < kChunk) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = -x[j];
          } else {   // q~ row (row - 64), columns c0 .. c0 + 15: two swizzled 16-byte chunks
            const int qi = row - kChunk;
            const unsigned char *qrow = sm + Lay::qt + (uint32_t)(c0 >> 6) * Lay::kPanel64 + (uint32_t)qi * 128;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
              const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + (((((c0 & 63) >> 3) + hc) ^ (qi & 7)) << 4));
              const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(h2[e]);
                x[8 * hc + 2 * e] = f.x - x[8 * hc + 2 * e];
                x[8 * hc + 2 * e + 1] = f.y - x[8 * hc + 2 * e + 1];
              }
            }
          }
          const uint32_t pan = Lay::WQ + (uint32_t)(c0 >> 6) * (128 * 128);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint4 w;
            w.x = pack_half2(x[8 * hc + 0], x[8 * hc + 1]);
            w.y = pack_half2(x[8 * hc + 2], x[8 * hc + 3]);
            w.z = pack_half2(x[8 * hc + 4], x[8 * hc + 5]);
            w.w = pack_half2(x[8 * hc + 6], x[8 * hc + 7]);
            *reinterpret_cast<uint4 *>(sm + pan + umma::sw128_chunk(row, ((c0 & 63) >> 3) + hc)) = w;
          }
        }
      }
      // The k~ buffer of chunk n + 1 was read by D3 of chunk n - 1. Observe that product before
      // releasing chunk n: afterwards the chain can run ahead and complete another phase.
      if (n > 0) wait_bar(&ms.bar_mma2, par ^ 1u);
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarPrep, kPrepGroupThreads);   // WQ complete; q~ consumed
      if (pt == 0 && !bad) {
        umma::mbar_arrive(&ms.bar_wq_full);
        if (n + 1 < nch) stage_q(n + 1);
      }
    }
  }

  // ---- exit: no bulk copy or tensor-core work of this CTA may be in flight past this point.
  // On a normal exit every copy was waited for; after a timeout, wait (bounded) for the
  // phases that were still open.
  if (tid == 0 || pt == 0) umma::commit(&ms.bar_exit);   // arrives once this thread's MMAs are done
  umma::mbar_wait_bounded(&ms.bar_exit, 0, kWaitLimit);
  if (!is_chain && *(volatile int *)&ms.err != 0) {
    // a copy issued for a chunk that was never processed may still be landing: wait for the
    // next phase of each copy barrier (returns at once if it completes, gives up otherwise)
    umma::mbar_wait_bounded(&ms.bar_in, in_done & 1u, kWaitLimit);
    umma::mbar_wait_bounded(&ms.bar_q, q_done & 1u, kWaitLimit);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (ms.err) {
    if (tid == 0) atomicExch(p.dev_status, kDevWaitTimeout);
  } else if (is_chain && p.final_state && tid < K) {
#pragma unroll
    for (int v = 0; v < kBV; ++v) p.final_state[(((long long)s * p.H + h) * p.V + v0 + v) * K + tid] = S[v];
  }
  if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <int K>
static cudaError_t launch_recur_t(const Problem &p, const TmaMaps &maps, cudaStream_t stream) {
  const size_t smem = RecLayout<K>::bytes;
  static_assert(sizeof(RecMisc<K>) <= 4096, "misc block");
  cudaError_t e = cudaFuncSetAttribute(recur_tc_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.H * (p.V / kBV);
  recur_tc_kernel<K><<<(unsigned)grid, kRecThreads, smem, stream>>>(p, maps);
  return cudaGetLastError();
}

cudaError_t launch_recur(const Problem &p, const TmaMaps &maps, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  return p.K == 64 ? launch_recur_t<64>(p, maps, stream) : launch_recur_t<128>(p, maps, stream);
}

}  // namespace kda
