// K2: head-parallel chunk recurrence of the KDA chunked forward, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, head, BV-wide slice of V; BV = 64, or 16 when that
// gives too few CTAs to fill the GPU). The CTA walks the chunks of its sequence
// in order and carries its K x BV slice of the state S (the
// FlashKDA "K2" stage, FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의
// 분리"; the cuLA "chunk gated delta h" + "chunk fwd o" stages, cuLA launch
// blog, section "Status & Roadmap"). Per chunk, with M = [-Tb ; P Tb] from
// the prep kernel and the in-chunk decays measured from the chunk start:
//
//   D1 = M (khat Gamma)          = [-w ; P w]        (128 x K,  UMMA 128xKx64)
//   D2 = M v                     = [-u ; P u]        (128 x BV, UMMA 128xBVx64)
//   WQ = [w ; q~ - P w],  q~ = qhat Gamma            (fp16 operand)
//   D2 += WQ S                   = [-U ; O]          (UMMA 128xBVxK)
//   U -> fp16, o = O -> bf16   (the output scale is folded into P and q~)
//   D3 = k~^T U,  k~ = khat Gamma_last / Gamma       (UMMA 128xBVx64)
//   S  = Gamma_last S + D3                           (fp32 master in registers)
//
// Gamma_i is the product of the per-token decays alpha up to token i (all
// factors <= 1, formed as products, never as quotients). U holds the
// delta-rule residuals v - prediction of the chunk; O the inter-chunk term
// q~ S plus the intra-chunk term P U.
//
// The prep kernel hands over M, khat Gamma and k~ (as swizzled operand images),
// q~ and Gamma_last per chunk; v comes straight from the input by TMA. D1 and D2 are
// one product M [khat Gamma | v], and WQ is written to tensor memory, where MMA1
// reads its A operand: shared-memory bandwidth, which every tcgen05.mma operand
// and every staged copy shares, bounds this kernel.
//
// Warp roles:
//   chain, warps 0-3: D2 += WQ S, U and o, D3 = k~^T U, S update, chunk after chunk.
//   two prep sub-groups, warps 4-7 (even chunks) and 8-11 (odd chunks): each stages its chunks'
//     operands (bulk copies and one TMA tile of v), converts v to fp16, issues D12 and forms WQ
//     into tensor memory. A sub-group has two chunk periods for each of its chunks, so the
//     S-independent work stays off the chain's path.
// Every buffer and barrier the sub-groups use exists once per chunk parity; each mbarrier
// carries one phase per chunk of its parity and a new phase can only start after the previous
// one was waited for, so no wait can mistake one phase for another. Every wait gives up after a
// bounded time; the groups then agree (barrier with OR-reduction) to stop, drain their
// tensor-core work and copies, free TMEM and report KDA_DEVICE_WAIT_TIMEOUT.
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kChainThreads = 128;
constexpr int kSubThreads = 128;                              // one prep sub-group
constexpr int kRecThreads = kChainThreads + 2 * kSubThreads;
// V slice per CTA: 64 columns, or 16 when 64-column slices would leave most SMs idle (few long
// sequences); the operand panels keep their 64-column rows and a narrow slice uses their first
// columns.
constexpr int kBVWide = 64, kBVNarrow = 16;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clocks per wait
// named barrier ids (0 is __syncthreads): the chain, prep sub-groups 0 and 1, and the chain's U
// rows written
constexpr int kBarChain = 1, kBarE = 4;
__device__ __forceinline__ int sub_bar(int sg) { return 2 + sg; }

template <int K, int BV>
struct RecLayout {
  // byte offsets from the 1024-aligned dynamic shared memory base
  static constexpr uint32_t kPanel64 = 64 * 128;                 // 64 rows x 128 B
  // per chunk parity: [M (128 x 64 K-major, A of D12) | khat Gamma | v (fp16)]: khat Gamma
  // (64 x K) and v (64 x 64) are consecutive MN-major panels, the B operand of
  // D12 = M [khat Gamma | v]
  static constexpr uint32_t mk = 0;
  static constexpr uint32_t mk_kg = 128 * 128, mk_vh = mk_kg + (K / 64) * kPanel64, mk_size = mk_vh + kPanel64;
  static constexpr uint32_t Sh = mk + 2 * mk_size;               // K x 64    MN-major (B of MMA1)
  static constexpr uint32_t Uh = Sh + K * 128;                   // 64 x 64   MN-major (B of MMA2)
  static constexpr uint32_t rv = Uh + kPanel64;                  // per parity: bf16 v [64][BV]
  static constexpr uint32_t qt = rv + 2 * 64 * BV * 2;           // per parity: q~ image (64 x K)
  // per parity: [k~ (64 x 128 MN-major, A of MMA2) | Gamma_last (K fp32)]
  static constexpr uint32_t kb = qt + 2 * 128 * K;
  static constexpr uint32_t kb_gam = 2 * kPanel64;
  static constexpr uint32_t kb_size = (kb_gam + 4 * K + 1023) / 1024 * 1024;
  static constexpr uint32_t misc = kb + 2 * kb_size;
  static constexpr uint32_t bytes = misc + 1024 + 1024;          // + misc + alignment slack
};

// Tensor memory columns: D12 = [D1 | D2] of chunk parity b at b (K + 64). D2 accumulates the
// chain's WQ S; once D1 is read, WQ (fp16 pairs, the A operand of MMA1) replaces its first
// K / 2 columns. D3 follows both.
template <int K, int BV>
struct RecTmem {
  static constexpr uint32_t d12 = K + BV;
  static constexpr uint32_t d3 = 2 * d12;
  static_assert(d3 + BV <= 512, "tensor memory columns");
};

// Small per-CTA state after the operand buffers. Arrays of two are per chunk parity.
struct RecMisc {
  uint64_t bar_in[2], bar_qt[2], bar_kt[2], bar_d12[2], bar_wq[2], bar_mma2[2], bar_mma1[2], bar_o[2], bar_uh,
      bar_exit;
  uint32_t tmem_slot;
  int err;
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// MODE selects what one CTA computes (context parallelism, kda_cp.cu, for the two passes):
//   kPlain      (sequence, head, V slice): the whole sequence from its initial state.
//   kSegLocal   (sequence, segment g < n_seg - 1, head, slice of [V | K]): segment g from a zero
//               state (g > 0) or from the initial state (g = 0, value columns only). Columns
//               V + j carry the transition: start column e_j, v = 0. o is written for g = 0
//               only; the end state goes to seg_state.
//   kSegFinal   (sequence, segment g >= 1, head, V slice): segment g from its true start state
//               (seg_start), writing o, and the final state for the last segment.
constexpr int kPlain = 0, kSegLocal = 1, kSegFinal = 2;

template <int K, int BV, int MODE>
__global__ void __launch_bounds__(kRecThreads, 1)
recur_tc_kernel(const Problem p, const __grid_constant__ TmaMaps maps) {
  using Lay = RecLayout<K, BV>;
  using Tm = RecTmem<K, BV>;
  constexpr int CW = BV >= 32 ? 32 : 16;   // TMEM columns read per wait in the chain
  // With 64-column slices the prep sub-group that owns chunk n, idle until D3 of chunk n is done,
  // reads and converts U columns 32..63 of that chunk while the chain does columns 0..31.
  constexpr bool kHelpU = (BV == 64);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  RecMisc &ms = *reinterpret_cast<RecMisc *>(sm + Lay::misc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // column slices: of V, or of [V | K] in the segment-local pass
  const int VT = (MODE == kSegLocal ? p.V + K : p.V) / BV;
  const int bid = blockIdx.x;
  const int h = (bid / VT) % p.H;
  const int v0 = (bid % VT) * BV;   // first column of the slice
  int r = bid / (p.H * VT), seg = 0;
  if constexpr (MODE != kPlain) {   // r = sequence * (n_seg - 1) + (segment index within the pass)
    seg = r % (p.n_seg - 1) + (MODE == kSegFinal ? 1 : 0);
    r /= p.n_seg - 1;
  }
  // transition columns (segment-local pass, v0 >= V): v = 0 and the start state is the identity
  const bool trans = MODE == kSegLocal && v0 >= p.V;
  if (MODE == kSegLocal && trans && seg == 0) return;   // segment 0 starts from a known state
  pdl_wait();   // the prep kernel (when launched to overlap it) has finished and its writes are visible
  if (p.flag && *p.flag != kDevOk) return;
  const int s = p.cu ? p.order[r] : r;
  SeqInfo si = seq_info(p, s);
  if constexpr (MODE != kPlain) {   // the CTA's segment of the sequence
    int lo, hi;
    segment_chunks((si.len + kChunk - 1) / kChunk, seg, p.n_seg, lo, hi);
    si.t0 += lo * kChunk;
    si.chunk0 += lo;
    si.len = max(0, min(si.len - lo * kChunk, (hi - lo) * kChunk));
  }
  // o is written by the plain kernel, the final pass and segment 0 of the local pass
  const bool write_o = MODE != kSegLocal || seg == 0;
  // fp32 [.][cols][K] segment state block of (sequence, segment, head), cols = V + K or V
  auto seg_block = [&](float *base, int cols) -> float * {
    return base + (((long long)s * p.n_seg + seg) * p.H + h) * (long long)cols * K;
  };
  const uint32_t sbase = umma::smem_u32(sm);
  const int nch = (si.len + kChunk - 1) / kChunk;
  const bool is_chain = warp < 4;
  const int sg = is_chain ? 0 : (warp - 4) >> 2;   // prep sub-group (its chunk parity)
  const int lt = (tid - kChainThreads) & (kSubThreads - 1);   // thread within the sub-group

  // ---- set-up: zero the k~ operands (rows >= K stay zero when K = 64), TMEM, barriers
  for (int b = 0; b < 2; ++b)
    for (int x = tid; x < (int)(2 * Lay::kPanel64 / 16); x += kRecThreads)
      reinterpret_cast<uint4 *>(sm + Lay::kb + b * Lay::kb_size)[x] = make_uint4(0, 0, 0, 0);
  if (trans)   // v = 0 in transition columns: the fp16 v panels are zeroed once and never converted
    for (int b = 0; b < 2; ++b)
      for (int x = tid; x < (int)(Lay::kPanel64 / 16); x += kRecThreads)
        reinterpret_cast<uint4 *>(sm + Lay::mk + b * Lay::mk_size + Lay::mk_vh)[x] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      umma::mbar_init(&ms.bar_in[b], 1);
      umma::mbar_init(&ms.bar_qt[b], 1);
      umma::mbar_init(&ms.bar_kt[b], 1);
      umma::mbar_init(&ms.bar_d12[b], 1);
      umma::mbar_init(&ms.bar_wq[b], 1);
      umma::mbar_init(&ms.bar_mma2[b], 1);
      umma::mbar_init(&ms.bar_mma1[b], 1);
      umma::mbar_init(&ms.bar_o[b], kChainThreads - kChunk);   // the chain's O-row threads
    }
    umma::mbar_init(&ms.bar_uh, kSubThreads / 2);   // the two U-lane warps of a prep sub-group
    umma::mbar_init(&ms.bar_exit, 3);   // the three threads that issue tensor-core work
    umma::mbar_fence_init();
    ms.err = 0;
  }
  // Copies of chunk n, into the buffers of parity n & 1, issued by thread 0 of the sub-group that
  // owns the chunk (hand-off block of its (chunk, head) slot; v by TMA, tokens past T read as
  // zeros, tokens of the next packed sequence are zeroed after arrival):
  //   bar_in: [M | khat Gamma] and the v tile   consumed by D12 and the v conversion
  //   bar_qt: q~                                consumed by the WQ rows
  //   bar_kt: [k~ | Gamma_last]                 consumed by D3 and the state update
  auto slot_of = [&](int n) -> const unsigned char * {
    return p.hand + (((long long)si.chunk0 + n) * p.H + h) * p.hand_stride;
  };
  auto stage_in = [&](int n) {
    const int b = n & 1;
    static_assert(Lay::mk_kg == hand_off_kg(K), "input buffer layout");
    umma::mbar_arrive_expect_tx(&ms.bar_in[b], (uint32_t)(hand_off_qt(K) + (trans ? 0 : kChunk * BV * 2)));
    umma::bulk_g2s(sm + Lay::mk + b * Lay::mk_size, slot_of(n), (uint32_t)hand_off_qt(K), &ms.bar_in[b]);
    if (!trans)
      umma::tma_load_4d(sm + Lay::rv + b * (kChunk * BV * 2), &maps.v, v0, h, si.t0 + n * kChunk, si.b,
                        &ms.bar_in[b]);
  };
  auto stage_qt = [&](int n) {
    const int b = n & 1;
    umma::mbar_arrive_expect_tx(&ms.bar_qt[b], kChunk * K * 2);
    umma::bulk_g2s(sm + Lay::qt + b * (128 * K), slot_of(n) + hand_off_qt(K), kChunk * K * 2, &ms.bar_qt[b]);
  };
  auto stage_kt = [&](int n) {
    const int b = n & 1;
    unsigned char *kb = sm + Lay::kb + b * Lay::kb_size;
    umma::mbar_arrive_expect_tx(&ms.bar_kt[b], kChunk * K * 2 + K * 4);
    if constexpr (K == 128) {   // the smem buffer has the global block's internal offsets
      static_assert(Lay::kb_gam == hand_off_gam(K) - hand_off_kt(K), "chunk buffer layout");
      umma::bulk_g2s(kb, slot_of(n) + hand_off_kt(K), (uint32_t)(hand_off_gam(K) + 4 * K - hand_off_kt(K)),
                     &ms.bar_kt[b]);
    } else {
      umma::bulk_g2s(kb, slot_of(n) + hand_off_kt(K), kChunk * K * 2, &ms.bar_kt[b]);
      umma::bulk_g2s(kb + Lay::kb_gam, slot_of(n) + hand_off_gam(K), K * 4, &ms.bar_kt[b]);
    }
  };
  // barriers initialised and the zeroed operands ordered before the first copies, which start at
  // once: chunk 0 before the initial state is loaded
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (!is_chain && lt == 0 && sg == 0 && nch > 0) {
    stage_in(0);
    stage_qt(0);
    stage_kt(0);
  }
  // chain threads: state master S[k][0:BV] (fp32, thread k) and its fp16 operand copy
  // (element index of S[tid][v0 + v] = st0 + v * stv in either state layout)
  const int stv = (p.flags & kStateKV) ? 1 : K;
  float S[BV];
  if (is_chain && tid < K) {
    if (MODE == kPlain || (MODE == kSegLocal && seg == 0)) {
      const long long st0 = state_index(p, s, h, tid, v0);
#pragma unroll
      for (int v = 0; v < BV; ++v) S[v] = p.init ? state_load(p, st0 + v * stv) : 0.f;
    } else if (MODE == kSegLocal) {   // zero value columns, identity transition columns
#pragma unroll
      for (int v = 0; v < BV; ++v) S[v] = (trans && tid == v0 - p.V + v) ? 1.f : 0.f;
    } else {   // the segment's true start state from the combine
      const float *src = seg_block(p.seg_start, p.V) + (long long)v0 * K + tid;
#pragma unroll
      for (int v = 0; v < BV; ++v) S[v] = src[(long long)v * K];
    }
#pragma unroll
    for (int c = 0; c < BV / 8; ++c) {
      uint4 w;
      w.x = pack_half2(S[8 * c + 0], S[8 * c + 1]);
      w.y = pack_half2(S[8 * c + 2], S[8 * c + 3]);
      w.z = pack_half2(S[8 * c + 4], S[8 * c + 5]);
      w.w = pack_half2(S[8 * c + 6], S[8 * c + 7]);
      *reinterpret_cast<uint4 *>(sm + Lay::Sh + umma::sw128_chunk(tid, c)) = w;
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  // chunk 1 once chunk 0's inputs have landed, so that the first chunk has the memory to itself
  if (!is_chain && lt == 0 && sg == 1 && nch > 1) {
    if (umma::mbar_wait_bounded(&ms.bar_in[0], 0, kWaitLimit)) {
      stage_in(1);
      stage_qt(1);
      stage_kt(1);
    } else {
      atomicExch(&ms.err, 1);
    }
  }
  const uint32_t tmem = ms.tmem_slot;
  const uint32_t tD3 = tmem + Tm::d3;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool bad = false;   // this thread saw a wait time out
  // completed phases of this sub-group's copy barriers (for the drain after an error)
  uint32_t in_done = 0, qt_done = 0, kt_done = 0;

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
    // ======================= chain =======================
    bool stop = false;   // uniform over the chain (decided by the barrier reduction ending each chunk)
    for (int n = 0; n < nch && !stop; ++n) {
      const int b = n & 1;
      const uint32_t ph = (uint32_t)((n >> 1) & 1);
      const uint32_t tD12 = tmem + Tm::d12 * b, tD2 = tD12 + K;
      const unsigned char *kb = sm + Lay::kb + b * Lay::kb_size;
      const int t0 = si.t0 + n * kChunk;
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_wq[b], ph);
      const float gam = (tid < K) ? reinterpret_cast<const float *>(kb + Lay::kb_gam)[tid] : 0.f;
      if (tid == 0 && !bad) {   // D2 += WQ S  ->  [-U ; O]; WQ (A operand) in tensor memory
        const uint32_t id = umma::idesc_f16(128, BV, 0, 1);
        const uint64_t b0 = umma::sdesc_sw128(sbase + Lay::Sh, K * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks) umma::mma_f16_ts(tD2, tD12 + ks * 8, umma::desc_add(b0, ks * 2048), id, 1);
        umma::commit(&ms.bar_mma1[b]);
      }
      wait_bar(&ms.bar_mma1[b], ph);
      // U (rows < 64) -> fp16 operand; o = O (rows >= 64, the scale is folded into P and q~) ->
      // bf16 global. D3 = k~^T U needs U complete (the U warps meet at kBarE). The O warps' reads
      // of D2 only have to end before D12 of chunk n + 2 overwrites it: they arrive on bar_o of
      // this parity, which the prep sub-group waits for before that D12.
      const int c_end = (kHelpU && tid < kChunk) ? 32 : BV;   // U columns past 32: the prep sub-group
#pragma unroll 1
      for (int c0 = 0; c0 < c_end; c0 += CW) {
        float x[CW];
        if constexpr (CW == 32) umma::tmem_ld32(tD2 + lane_base + c0, x);
        else umma::tmem_ld16(tD2 + lane_base + c0, x);
        umma::tmem_ld_wait();
        if (tid >= kChunk && c0 + CW >= BV) {
          umma::fence_before_sync();
          umma::mbar_arrive(&ms.bar_o[b]);
        }
        if (tid < kChunk) {
#pragma unroll
          for (int hc = 0; hc < CW / 8; ++hc) {
            uint4 w;
            w.x = pack_half2(-x[8 * hc + 0], -x[8 * hc + 1]);
            w.y = pack_half2(-x[8 * hc + 2], -x[8 * hc + 3]);
            w.z = pack_half2(-x[8 * hc + 4], -x[8 * hc + 5]);
            w.w = pack_half2(-x[8 * hc + 6], -x[8 * hc + 7]);
            *reinterpret_cast<uint4 *>(sm + Lay::Uh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
          }
        } else if (tid - kChunk < L && !bad && write_o) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.o + tok_row(p, si.b, t0 + tid - kChunk, h) * p.V + v0 + c0);
#pragma unroll
          for (int hc = 0; hc < CW / 8; ++hc) {
            __nv_bfloat16 ob[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) ob[j] = __float2bfloat16_rn(x[8 * hc + j]);
            dst[hc] = *reinterpret_cast<const uint4 *>(ob);
          }
        }
      }
      if (tid < kChunk) {
        umma::fence_proxy_async_smem();
        umma::fence_before_sync();
        umma::named_bar(kBarE, kChunk);
      }
      if (kHelpU && tid == 0) wait_bar(&ms.bar_uh, (uint32_t)(n & 1));   // the sub-group's U columns
      if (tid == 0 && !bad) {   // D3 = k~^T U
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, BV, 1, 1);
        const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::kb + b * Lay::kb_size, Lay::kPanel64, 1024);
        const uint64_t b0 = umma::sdesc_sw128(sbase + Lay::Uh, Lay::kPanel64, 1024);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tD3, umma::desc_add(a0, ks * 2048), umma::desc_add(b0, ks * 2048), id, ks > 0);
        umma::commit(&ms.bar_mma2[b]);
      }
      wait_bar(&ms.bar_mma2[b], ph);
      // S = gamma S + D3 (thread = channel), fp16 copy for the next chunk
      if (tid < K) {
#pragma unroll
        for (int c0 = 0; c0 < BV; c0 += CW) {
          float x[CW];
          if constexpr (CW == 32) umma::tmem_ld32(tD3 + lane_base + c0, x);
          else umma::tmem_ld16(tD3 + lane_base + c0, x);
          umma::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CW; ++j) S[c0 + j] = fmaf(gam, S[c0 + j], x[j]);
#pragma unroll
          for (int hc = 0; hc < CW / 8; ++hc) {
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
      // Sh complete; also the chain's agreement to stop after an error
      stop = umma::bar_red_or(kBarChain, kChainThreads, bad || *(volatile int *)&ms.err != 0);
    }
  } else {
    // ======================= prep sub-group sg: chunks n = sg, sg + 2, ... =======================
    const int b = sg;
    const uint32_t tD12 = tmem + Tm::d12 * b;
    unsigned char *mkb = sm + Lay::mk + b * Lay::mk_size;
    __nv_bfloat16 *rvb = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rv + b * (kChunk * BV * 2));
    const unsigned char *qtb = sm + Lay::qt + b * (128 * K);
    const int row = (warp & 3) * 32 + lane;   // TMEM lane of this warp's quadrant
    // U columns 32..63 of chunk m of this parity (the U-lane warps, after MMA1 of chunk m): fp16
    // into the operand of D3, then an arrival the chain's D3 issue waits for. The arrival also
    // comes after an error, so that the chain's bounded wait is only the last resort. MMA1 has a
    // barrier per chunk parity: this sub-group has waited for the phase of chunk m - 2, and the
    // phase of chunk m + 2 needs its own work of chunk m + 2, so the wait cannot alias.
    auto help_u = [&](int m) {
      if (!kHelpU || (warp & 3) >= 2) return;
      wait_bar(&ms.bar_mma1[b], (uint32_t)((m >> 1) & 1));
      if (!bad) {
        float x[32];
        umma::tmem_ld32(tD12 + K + lane_base + 32, x);
        umma::tmem_ld_wait();
#pragma unroll
        for (int hc = 0; hc < 4; ++hc) {
          uint4 w;
          w.x = pack_half2(-x[8 * hc + 0], -x[8 * hc + 1]);
          w.y = pack_half2(-x[8 * hc + 2], -x[8 * hc + 3]);
          w.z = pack_half2(-x[8 * hc + 4], -x[8 * hc + 5]);
          w.w = pack_half2(-x[8 * hc + 6], -x[8 * hc + 7]);
          *reinterpret_cast<uint4 *>(sm + Lay::Uh + umma::sw128_chunk(row, 4 + hc)) = w;
        }
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::mbar_arrive(&ms.bar_uh);
    };
    int pending = -1;   // the last chunk of this sub-group whose U columns are still to be done
    for (int n = sg; n < nch; n += 2) {
      const uint32_t ph = (uint32_t)((n >> 1) & 1);
      const int L = min(kChunk, si.len - n * kChunk);
      if (n >= 2) help_u(n - 2);
      pending = -1;
      // -- v of chunk n -> fp16, the panel after khat Gamma (vh was last read by D12 of chunk n - 2)
      wait_bar(&ms.bar_in[b], ph);
      in_done += bad ? 0u : 1u;
      if (!trans && L < kChunk) {   // v rows past the sequence end (next packed sequence or zero fill): zero them
        for (int x = lt; x < (kChunk - L) * (BV / 8); x += kSubThreads) {
          const int i = L + x / (BV / 8), c8 = x % (BV / 8);
          *reinterpret_cast<uint4 *>(rvb + i * BV + 8 * c8) = make_uint4(0, 0, 0, 0);
        }
        umma::named_bar(sub_bar(sg), kSubThreads);
      }
#pragma unroll
      for (int j = 0; j < (trans ? 0 : kChunk * BV / 8 / kSubThreads); ++j) {   // 16-byte chunks of the tile
        const int x = lt + kSubThreads * j;
        const int i = x / (BV / 8), cc = x % (BV / 8);
        const uint4 raw = *reinterpret_cast<const uint4 *>(rvb + i * BV + 8 * cc);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
        const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
        *reinterpret_cast<uint4 *>(mkb + Lay::mk_vh + umma::sw128_chunk(i, cc)) =
            make_uint4(pack_half2(f0.x, f0.y), pack_half2(f1.x, f1.y), pack_half2(f2.x, f2.y),
                       pack_half2(f3.x, f3.y));
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      // vh complete, the v tile consumed; also the sub-group's agreement to stop after an error
      if (umma::bar_red_or(sub_bar(sg), kSubThreads, bad || *(volatile int *)&ms.err != 0)) break;
      // -- D12 of chunk n overwrites the accumulators, WQ and k~ buffer of chunk n - 2: wait for D3
      //    of chunk n - 2 (after it the chain has read them all). The next phase of that barrier
      //    (chunk n) needs WQ of chunk n, so this wait cannot see the wrong phase.
      if (n >= 2) {
        wait_bar(&ms.bar_mma2[b], (uint32_t)(((n - 2) >> 1) & 1));
        wait_bar(&ms.bar_o[b], (uint32_t)(((n - 2) >> 1) & 1));   // and the chain's O rows of chunk n - 2 read
      }
      if (lt == 0 && !bad) {
        if (n >= 2) stage_kt(n);
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, K + BV, 0, 1);   // D12 = M [khat Gamma | v]
        const uint64_t a0 = umma::sdesc_sw128(umma::smem_u32(mkb), 16, 1024);
        const uint64_t b0 = umma::sdesc_sw128(umma::smem_u32(mkb + Lay::mk_kg), Lay::kPanel64, 1024);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tD12, umma::desc_add(a0, ks * 32), umma::desc_add(b0, ks * 2048), id, ks > 0);
        umma::commit(&ms.bar_d12[b]);
      }
      wait_bar(&ms.bar_d12[b], ph);
      if (lt == 0 && !bad && n + 2 < nch) stage_in(n + 2);   // M, khat Gamma, v of chunk n are consumed
      wait_bar(&ms.bar_qt[b], ph);
      qt_done += bad ? 0u : 1u;
      // -- WQ rows: w = -D1 (rows < 64), q~ - D1 (rows >= 64), as fp16 pairs over the first K / 2
      //    columns of D1. This warp owns its 32 lanes. Step t reads D1 columns [32 t, 32 t + 32) and
      //    writes WQ columns [16 t, 16 t + 16), which step t / 2 <= t has already read.
#pragma unroll 1
      for (int c0 = 0; c0 < K; c0 += 32) {
        float x[32];
        umma::tmem_ld32(tD12 + lane_base + c0, x);
        umma::tmem_ld_wait();
        if (row < kChunk) {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = -x[j];
        } else {   // q~ row (row - 64), columns c0 .. c0 + 31: four swizzled 16-byte chunks
          const int qi = row - kChunk;
          const unsigned char *qrow = qtb + (uint32_t)(c0 >> 6) * Lay::kPanel64 + (uint32_t)qi * 128;
#pragma unroll
          for (int hc = 0; hc < 4; ++hc) {
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
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) pk[j] = pack_half2(x[16 * hs + 2 * j], x[16 * hs + 2 * j + 1]);
          umma::tmem_st8(tD12 + lane_base + (uint32_t)((c0 + 16 * hs) >> 1), pk);
        }
      }
      umma::tmem_st_wait();
      umma::fence_proxy_async_smem();   // q~ reads before the bulk copy that reuses the buffer
      umma::fence_before_sync();
      umma::named_bar(sub_bar(sg), kSubThreads);   // WQ complete; q~ consumed
      if (lt == 0 && !bad && n + 2 < nch) stage_qt(n + 2);
      wait_bar(&ms.bar_kt[b], ph);   // k~ and Gamma_last of chunk n landed
      kt_done += bad ? 0u : 1u;
      if (lt == 0 && !bad) umma::mbar_arrive(&ms.bar_wq[b]);
      pending = n;
    }
    if (pending >= 0) help_u(pending);
  }

  // ---- exit: no bulk copy or tensor-core work of this CTA may be in flight past this point.
  // On a normal exit every copy was waited for; after a timeout, wait (bounded) for the
  // phases that were still open.
  if (tid == 0 || (!is_chain && lt == 0)) umma::commit(&ms.bar_exit);   // arrives once its MMAs are done
  umma::mbar_wait_bounded(&ms.bar_exit, 0, kWaitLimit);
  if (!is_chain && *(volatile int *)&ms.err != 0) {
    // a copy issued for a chunk that was never processed may still be landing: wait for the
    // next phase of each of this sub-group's copy barriers (returns at once if it completes,
    // gives up otherwise)
    umma::mbar_wait_bounded(&ms.bar_in[sg], in_done & 1u, kWaitLimit);
    umma::mbar_wait_bounded(&ms.bar_qt[sg], qt_done & 1u, kWaitLimit);
    umma::mbar_wait_bounded(&ms.bar_kt[sg], kt_done & 1u, kWaitLimit);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (ms.err) {
    if (tid == 0) atomicExch(p.dev_status, kDevWaitTimeout);
  } else if (is_chain && tid < K) {
    // An fp16 overflow of S, U or v (or a non-finite input) leaves inf / NaN in the fp32 state,
    // which keeps it to the end: one look at the last state reports it (whole warps take part).
    bool finite = true;
#pragma unroll
    for (int v = 0; v < BV; ++v) finite &= fabsf(S[v]) <= 3.402823466e38f;
    if (__any_sync(0xffffffffu, !finite) && lane == 0) atomicExch(p.dev_status, kDevNonFinite);
    if (MODE == kSegLocal) {   // end state of the segment (or its transition) for the combine
      float *dst = seg_block(p.seg_state, p.V + K) + (long long)v0 * K + tid;
#pragma unroll
      for (int v = 0; v < BV; ++v) dst[(long long)v * K] = S[v];
    } else if (p.final_state && (MODE == kPlain || seg == p.n_seg - 1)) {
#pragma unroll
      for (int v = 0; v < BV; ++v) state_store(p, state_index(p, s, h, tid, v0) + v * stv, S[v]);
    }
  }
  if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <int K, int BV, int MODE>
static cudaError_t launch_recur_t(const Problem &p, const TmaMaps &maps, cudaStream_t stream, bool overlap) {
  const size_t smem = RecLayout<K, BV>::bytes;
  static_assert(sizeof(RecMisc) <= 1024, "misc block");
  static PerDeviceOnce attr;
  cudaError_t e = attr([&](int) {
    return cudaFuncSetAttribute(recur_tc_kernel<K, BV, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
  });
  if (e != cudaSuccess) return e;
  const int cols = MODE == kSegLocal ? p.V + K : p.V;
  const long long jobs = MODE == kPlain ? (long long)p.N : (long long)p.N * (p.n_seg - 1);
  const long long grid = jobs * p.H * (cols / BV);
  return launch_kernel(recur_tc_kernel<K, BV, MODE>, dim3((unsigned)grid), dim3(kRecThreads), smem, stream,
                       overlap, p, maps);
}

// SM count of the current device (looked up once per device), or 0 if it cannot be read.
int device_sm_count() {
  static PerDeviceOnce once;
  static std::atomic<int> sm_count[64];
  int sms = 0;
  const cudaError_t e = once([&](int dev) {
    int n = 0;
    const cudaError_t r = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess && dev >= 0 && dev < 64) sm_count[dev].store(n, std::memory_order_relaxed);
    sms = n;
    return r;
  });
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (sms == 0) {   // looked up by an earlier call on this device
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms == 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  return sms;
}

// V-slice width: 64 unless that leaves fewer than about 80% of the SMs with a CTA.
int slice_width_for(long long N, int H, int V, int sms) {
  if (sms <= 0) return kBVWide;
  const long long wide_ctas = N * H * (V / kBVWide);
  return (5 * wide_ctas >= 4LL * sms) ? kBVWide : kBVNarrow;
}
int recur_slice_width(const Problem &p) { return slice_width_for(p.N, p.H, p.V, device_sm_count()); }

cudaError_t launch_recur(const Problem &p, const TmaMaps &maps, int bv, cudaStream_t stream, bool overlap) {
  if (p.N == 0) return cudaSuccess;
  if (bv == kBVNarrow)
    return p.K == 64 ? launch_recur_t<64, kBVNarrow, kPlain>(p, maps, stream, overlap)
                     : launch_recur_t<128, kBVNarrow, kPlain>(p, maps, stream, overlap);
  return p.K == 64 ? launch_recur_t<64, kBVWide, kPlain>(p, maps, stream, overlap)
                   : launch_recur_t<128, kBVWide, kPlain>(p, maps, stream, overlap);
}

// The two recurrence passes of context parallelism (64-column slices): pass 1 runs every segment
// but the last from a zero (or, for segment 0, the initial) state with the transition columns;
// pass 2 runs every segment but the first from the start state the combine formed.
cudaError_t launch_recur_segments(const Problem &p, const TmaMaps &maps, int pass, cudaStream_t stream,
                                  bool overlap) {
  if (p.N == 0 || p.n_seg < 2) return cudaSuccess;
  if (pass == 1)
    return p.K == 64 ? launch_recur_t<64, kBVWide, kSegLocal>(p, maps, stream, overlap)
                     : launch_recur_t<128, kBVWide, kSegLocal>(p, maps, stream, overlap);
  return p.K == 64 ? launch_recur_t<64, kBVWide, kSegFinal>(p, maps, stream, overlap)
                   : launch_recur_t<128, kBVWide, kSegFinal>(p, maps, stream, overlap);
}

}  // namespace kda
