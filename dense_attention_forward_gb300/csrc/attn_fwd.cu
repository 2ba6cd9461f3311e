// attn_fwd.cu -- fused dense attention forward for GB300 (sm_103a): kernel + C ABI.
//
// O = softmax(scale * Q K^T) V and the fp32 logsumexp for BF16 Q/K/V of shape [B, H, S, 128].
//
// Design (after "B200 attention kernel from scratch to ~SOTA in 60 figures (CUDA/PTX)",
// cited as [B200-attn]; its kernels were written for B200 and are prior art here):
//  * Work split (Ch. 1 §ii, Ch. 5): a work item is two consecutive 128-row Q tiles of one
//    (batch, head), walked against every 128-key K/V tile of that head; each K/V tile loaded
//    into shared memory serves both Q tiles. One CTA per SM walks a list of items (persistent
//    grid), so the next item's Q loads and first QK overlap the current item's last tiles and
//    epilogue instead of a CTA exit, launch and pipeline fill per item.
//  * Loads (Ch. 3, Ch. 6): Q0, K0 and Q1 leave right after the barriers are initialised; one
//    TMA warp then streams K and V as separate tokens through a kStages-slot ring of 32 KB
//    SW128 slots. A slot is refilled once the second Q tile's softmax warps have taken the S
//    that follows its last consumer (that tile's QK for K, its PV for V): they publish a
//    monotonic count of the S tiles they have taken, so no MMA commit is spent on freeing
//    slots and no parity wait can mistake one phase for another two steps away.
//  * MMA (Ch. 1 §A/§C, Ch. 2, Ch. 5, Ch. 7, Ch. 13): tcgen05.mma M128 N128 K16, S_q = Q_q K^T
//    (both K-major SW128 in shared memory) and O_q += P_q V (P from tensor memory, V MN-major
//    SW128). One warp per Q tile issues that tile's MMAs: in K/V tile i, the PV_q(i) steps of
//    each part of P_q(i) as soon as the softmax has stored that part (the pages' "early PV"),
//    then QK_q(i+1). The two issuing warps take turns group by group, so one Q tile's softmax
//    overlaps the other's MMAs (ping-pong).
//  * Softmax (Ch. 1 §B, Ch. 8, Ch. 11): 4 warps per Q tile, one thread per row, the whole
//    128-score row in registers; base-2 exponent with scale*log2(e) folded into one factor,
//    row max taken on raw scores; P is packed to BF16 pairs and stored over S in tensor
//    memory. The kept row max moves only when a tile's max exceeds it by the rebase threshold
//    (Ch. 11): 1 by default (P <= 2), 0 (the running max, P <= 1) or the pages' 8, with O then
//    normalised by the sum of the BF16-rounded P. Only packed FP32x2 arithmetic, MUFU,
//    conversions and byte permutes run per element: on this part scalar FP32 and IMAD work
//    in other warps slows the tensor pipe.
//  * Correction (Ch. 11, Ch. 12): 4 warps shared by both Q tiles rescale O in tensor memory
//    when any row of their 32 rebased.
//  * Epilogue (Ch. 1): each softmax warp reads its 32 rows of O out of tensor memory (which
//    frees O_q for the next item's first PV), turns O / l into BF16 and TMA-stores it from its
//    own 4 KB SW128 staging slice in two half-width passes (32-row boxes, no cross-warp
//    barrier); lse = (m + log2 l) * ln 2 is written by the same threads.
//
// Barrier phases count across the items of a CTA: per K/V tile of the CTA's stream (S full,
// O safe, the turns, the P parts), per item (Q full, O full) or per token (the K/V ring).
// TMEM: 512 columns = S0 [0,128) | S1 [128,256) | O0 [256,384) | O1 [384,512); P_q occupies
// the first 64 columns of S_q. Warps 0-7 softmax, 8-11 correction, 12 and 13 MMA issue (13
// also owns the TMEM allocation), 14 loads, 15 set-up (then idle, so that no working warp runs
// diverged set-up code). Every mbarrier wait is bounded (about two
// seconds); a CTA that gives up records the failure in a device status word, drains its own
// TMA loads and MMAs, frees its tensor memory and exits. The only other barriers are the
// CTA-wide ones at entry and exit, and the named barriers on which each Q tile's softmax warps
// (arriving) meet its issuing warp (waiting), one per part of P. Those have no timeout, so the
// softmax warps only ever arrive for a tile whose S they have seen, and wait for a tile's S
// until the issuing warp announces that it has stopped; the issuing warp only waits at a tile's
// barriers after issuing that tile's QK (see wait_s_full).
// The test-hook build (-DATTN_TEST_HOOKS, libattn_testhooks.so) adds attn_fwd_withhold, which
// runs this path on purpose: its producer skips one K/V token, so the waits on that token run
// out. The product build has neither that entry point nor the parameter.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "attn.h"
#ifdef ATTN_TEST_HOOKS
#include "attn_test_hooks.h"
#endif
#include "ptx.cuh"

namespace gb300 {

constexpr int kBlock = 128;                      // rows per Q tile and keys per K/V tile
constexpr int kHeadDim = 128;                    // D
constexpr int kTileBytes = kBlock * kHeadDim * 2;  // one 128x128 BF16 tile: 32 KB
constexpr int kSliceBytes = kBlock * 128;        // 128 rows x 128 B: one SW128 column of atoms
constexpr int kStages = 4;                       // K/V ring slots
constexpr int kThreads = 512;                    // 16 warps
constexpr int kLoadWarp = 14;                    // TMA producer
constexpr int kIssueWarp0 = 12;                  // MMA issue for Q tile 0
constexpr int kIssueWarp1 = 13;                  // MMA issue for Q tile 1; also owns the TMEM allocation
constexpr int kTmemWarp = kIssueWarp1;
constexpr int kSetupWarp = 15;                   // set-up (barriers, first loads); idle after
// P_q(i) is stored and consumed in parts: packed BF16 pairs (TMEM columns) [kPCut[k], kPCut[k+1]).
// A PV K16 step reads 8 of them, so every cut is a multiple of 8. A small first part lets the
// tensor pipe start PV_q(i) early; QK_q(i+1) waits for the last part.
constexpr int kPParts = 3;
constexpr int kPCut[kPParts + 1] = {0, 16, 40, 64};
constexpr int kBarP = 2;  // named barrier of part k of Q tile q: kBarP + 2k + q (0 is __syncthreads)
constexpr int kDefaultRebase = 1;                // rebase threshold of attn_fwd, attn_fwd_causal, attn_fwd_host
static_assert(kBarP + 2 * kPParts <= 16, "named barrier ids");
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;  // drain after a failure: 0.2 s
// The softmax warps' wait for S, bounded well beyond the issuing warp's worst case (its waits
// between two QK groups, each bounded by kWaitLimitNs; see wait_s_full).
constexpr uint64_t kSWaitLimitNs = 10000000000ull;

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;                                   // Q0, Q1
constexpr int kOffKV = kOffQ + 2 * kTileBytes;             // K/V ring
constexpr int kOffStage = kOffKV + kStages * kTileBytes;   // O staging: [2 tiles][4 warps] x 4 KB
constexpr int kStageWarpBytes = 32 * 128;                  // 32 rows x 64 columns of BF16
constexpr int kOffBar = kOffStage + 8 * kStageWarpBytes;   // mbarriers
// barrier indices
constexpr int kBarQFull = 0;                       // [2] Q_q landed (TMA bytes)
constexpr int kBarKVFull = 2;                      // [kStages] token landed (TMA bytes)
constexpr int kBarSFull = kBarKVFull + kStages;    // [2] S_q in TMEM (MMA commit)
constexpr int kBarOSafe = kBarSFull + 2;           // [2] O_q rescaled or left as is (4 correction warps)
constexpr int kBarOFull = kBarOSafe + 2;           // [2] last PV_q done (MMA commit)
constexpr int kBarStats = kBarOFull + 2;           // [2] per-row rescale factors published (4 warps)
constexpr int kBarMmaDone = kBarStats + 2;         // [2] drain after a failure (one per issuing warp)
constexpr int kBarTurn = kBarMmaDone + 2;          // [2] MMA-group turn of Q tile q (from the other issuing warp)
constexpr int kNumBars = kBarTurn + 2;
constexpr int kSeenCode = kNumBars;                // status-word index of the wait on S-seen count q: kSeenCode + q
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffFail = kOffAbort + 4;                    // int[2]: issuing warp q has stopped issuing
constexpr int kOffSeen = kOffFail + 8;                     // int[2]: S_q tiles seen by the softmax warps
constexpr int kOffAlpha = (kOffSeen + 8 + 15) & ~15;       // float[2][128]
constexpr int kMaxOrder = 384;                             // causal: most items a CTA sorts
constexpr int kOffOrder = kOffAlpha + 2 * kBlock * 4;      // uint16[kMaxOrder]: the CTA's causal item order
constexpr int kSmemUsed = kOffOrder + kMaxOrder * 2;
constexpr int kSmemBytes = kSmemUsed + 1024;               // slack for the 1024-byte alignment

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffKV % 1024 == 0 && kTileBytes % 1024 == 0, "SW128 atoms need 1024-B alignment");

// Failure codes written to the device status word: 0xA77E0000 | role << 8 | barrier index.
enum : uint32_t { kRoleLoad = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleCorrection = 4 };

__device__ unsigned int g_attn_status = 0;

// Optional timeline trace (built only into libattn_trace.so, with -DATTN_TRACE): per CTA, the
// globaltimer at entry (0), after setup (1), when Q tile 0's first S is seen (2), when O_0 and
// O_1 are full (3, 4), before the final barrier (5), the SM id (6) and at exit (7); and, at the
// boundary between the CTA's first two items, for Q tile 0: the first item's last S seen (8),
// its last P part stored (9), O read out of tensor memory (10), epilogue done (11), the next
// item's first S seen (12) and first P part stored (13), and by the issuing warp the next
// item's first QK issued (14) and first PV issued (15). In the ordinary build the stamps
// compile to nothing.
#ifdef ATTN_TRACE
#ifndef ATTN_TRACE_CTAS
#define ATTN_TRACE_CTAS 4096
#endif
constexpr int kTraceWords = 16;  // per CTA
__device__ unsigned long long g_attn_trace[ATTN_TRACE_CTAS * kTraceWords];
__device__ __forceinline__ unsigned sm_id() {
  unsigned r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
#define ATTN_STAMP(k)                                                                        \
  do {                                                                                       \
    if (blockIdx.x < ATTN_TRACE_CTAS) g_attn_trace[blockIdx.x * kTraceWords + (k)] = global_timer_ns(); \
  } while (0)
#define ATTN_STAMP_SM()                                                   \
  do {                                                                    \
    if (blockIdx.x < ATTN_TRACE_CTAS) g_attn_trace[blockIdx.x * kTraceWords + 6] = sm_id(); \
  } while (0)
// A stamp taken only when cond holds; outside the trace build neither is compiled.
#define ATTN_STAMP_IF(cond, k) \
  do {                          \
    if (cond) ATTN_STAMP(k);    \
  } while (0)
#else
#define ATTN_STAMP_IF(cond, k)
#define ATTN_STAMP(k) \
  do {                \
  } while (0)
#define ATTN_STAMP_SM() \
  do {                  \
  } while (0)
#endif

struct Params {
  float* lse;
  int S;            // sequence length
  int H;            // heads (the tensor maps are 4-D: {D, S, H, B})
  int n_kv;         // ceil(S / 128)
  int n_qp;         // ceil(S / 256): Q-tile pairs per (b, h)
  int BH;           // B * H
  int num_items;    // B * H * n_qp work items (a pair of Q tiles each)
  float scale_log2; // scale * log2(e)
#ifdef ATTN_TEST_HOOKS
  int withhold;     // K/V token the producer never loads (bounded-wait test hook), -1: none
#endif
};

// Whether the producer skips token t (only the test-hook build ever does).
#ifdef ATTN_TEST_HOOKS
#define ATTN_WITHHELD(p, t) ((t) == (p).withhold)
#else
#define ATTN_WITHHELD(p, t) false
#endif

struct Ctl {
  uint32_t bar0;                  // smem address of barrier 0
  volatile uint32_t* abort_flag;  // shared
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * i; }
};

__device__ __forceinline__ bool wait_slow(const Ctl& c, int b, uint32_t parity, uint32_t role,
                                          bool watch_abort, uint64_t limit_ns) {
  const uint32_t bar = c.bar(b);
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (watch_abort && *c.abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        if (watch_abort) {
          *c.abort_flag = 1u;
          atomicCAS(&g_attn_status, 0u, 0xA77E0000u | (role << 8) | static_cast<uint32_t>(b));
        }
        return false;
      }
    }
  }
}

// Wait for phase `parity` of barrier b; false if this CTA is giving up.
__device__ __forceinline__ bool wait_bar(const Ctl& c, int b, uint32_t parity, uint32_t role) {
  if (mbar_try_wait(c.bar(b), parity)) return true;
  return wait_slow(c, b, parity, role, true, kWaitLimitNs);
}

// Warp-uniform variant for code that continues with warp-collective tcgen05 instructions.
__device__ __forceinline__ bool wait_bar_warp(const Ctl& c, int b, uint32_t parity, uint32_t role) {
  const bool ok = wait_bar(c, b, parity, role);
  return __all_sync(0xffffffffu, ok);
}

// The softmax warps' wait for S_q full (warp-uniform result). It does not give up on the CTA's
// abort flag: it returns false only once the issuing warp has announced that it stopped issuing
// (*stopped), or after kSWaitLimitNs. The issuing warp waits at a tile's named barriers only
// after issuing that tile's QK, whose completion this wait always sees, so the softmax warps
// never leave those barriers short of their arrivals, and they never arrive at a barrier twice
// while the issuing warp has yet to pass it (a named barrier has no generations to tell the two
// apart).
__device__ __noinline__ bool wait_s_full_slow(uint32_t bar, uint32_t parity, volatile int* stopped,
                                              volatile uint32_t* abort_flag, uint32_t code) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*stopped) return false;
      if (global_timer_ns() - t0 > kSWaitLimitNs) {
        *abort_flag = 1u;
        atomicCAS(&g_attn_status, 0u, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_s_full(const Ctl& c, int b, uint32_t parity, volatile int* stopped) {
  bool ok = mbar_try_wait(c.bar(b), parity);
  if (!ok)
    ok = wait_s_full_slow(c.bar(b), parity, stopped, c.abort_flag,
                          0xA77E0000u | (kRoleSoftmax << 8) | static_cast<uint32_t>(b));
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int ld_acquire_shared(const volatile int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(const_cast<int*>(p))) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_shared(volatile int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(const_cast<int*>(p))), "r"(v) : "memory");
}

// The TMA producer's wait until *count >= target (a monotonic count, so unlike a parity wait it
// cannot mistake a phase two steps ahead or behind for the one it wants); false if this CTA is
// giving up.
__device__ __noinline__ bool wait_count(const Ctl& c, const volatile int* count, int target, uint32_t code) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_shared(count) >= target) return true;
    __nanosleep(32);
    if ((it & 15u) == 0) {
      if (*c.abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *c.abort_flag = 1u;
        atomicCAS(&g_attn_status, 0u, code);
        return false;
      }
    }
  }
}

// One arrival per warp, after every lane's prior shared/tensor-memory writes are ordered by
// __syncwarp (each lane has already fenced its tcgen05 stores where that matters).
__device__ __forceinline__ void warp_arrive(const Ctl& c, int b, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(c.bar(b));
}

// Arrival without waiting (the producer side of a named barrier).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Calls f(integral_constant<int, 0>) ... f(integral_constant<int, N - 1>): one body per part
// of P, with compile-time column ranges.
template <int N, int I = 0, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<N, I + 1>(f);
  }
}

// kThr: the rebase threshold of the pages' Ch. 11 "skip O rescale", in base-2 units. The kept
// row max moves (and O, l are rescaled) only when a tile's max exceeds it by kThr or more
// (threshold 0: whenever it grows, so the kept max is the running max). P then stays below
// 2^kThr. For 0 and 1 one fp32 row sum serves both O and lse: the BF16 rounding of P in the
// PV product against the fp32 sum is at most 2^-9 relative per term, which for P <= 2 stays
// well inside the output tolerance even on rows dominated by one key. For 8, P can reach 256
// and O is normalised by a second row sum over the BF16-rounded P.
// kCausal: query i sees keys j <= i (queries and keys share positions 0..S-1). The item of Q
// tiles 2qp and 2qp+1 walks K/V tiles 0..2qp+1 only; its diagonal tiles are masked per
// element, and Q tile 2qp runs tile 2qp+1 fully masked (P = 0) so both Q tiles keep the same
// K/V schedule. Items are dealt to the CTAs longest first in a snake order, which evens out
// the CTAs' totals of K/V tiles; each CTA then takes its items head by head (see sorted_order).
template <int kThr, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw_addr);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  // Work items are pairs of 128-row Q tiles of one (batch, head). CTA c takes the items of
  // rounds r = 0, 1, ...: dense, item r * gridDim.x + c (items are numbered head-major, so the
  // CTAs of one round share K/V in L2); causal, items sorted longest first across all heads and
  // dealt out in a snake (c, then 2 * gridDim.x - 1 - c, ...) so that every CTA gets a similar
  // total of K/V tiles (the CTA then takes its own items in head order, see sorted_order).
  const int item0 = static_cast<int>(blockIdx.x);
  const int stride = static_cast<int>(gridDim.x);
  auto item_of = [&](int r) {
    return (kCausal && (r & 1)) ? r * stride + stride - 1 - item0 : r * stride + item0;
  };
  struct Item {
    int qp, bh, hh, bb, q0, n;
  };
  // Items of this CTA: rounds r < n_mine (the rounds that exist form a prefix; the last, partial
  // round reaches the CTAs at positions below its size).
  const int full_rounds = p.num_items / stride;
  const int last_pos = (kCausal && (full_rounds & 1)) ? stride - 1 - item0 : item0;
  const int n_mine = full_rounds + (last_pos < p.num_items % stride ? 1 : 0);
  auto item_at = [&](int it) {
    Item r;
    if constexpr (kCausal) {
      r.qp = p.n_qp - 1 - it / p.BH;
      r.bh = it % p.BH;
    } else {
      r.qp = it % p.n_qp;
      r.bh = it / p.n_qp;
    }
    r.hh = r.bh % p.H;
    r.bb = r.bh / p.H;
    r.q0 = r.qp * 2 * kBlock;
    r.n = kCausal ? min(p.n_kv, 2 * r.qp + 2) : p.n_kv;
    return r;
  };

  // Causal: the snake sets which items a CTA holds (and so the balance); the CTA takes them by
  // (batch * head, longest first), so that at any moment the CTAs work on few heads and their
  // K/V tiles are read from DRAM about once instead of once per round. The order is sorted at
  // set-up into shared memory by the set-up warp; a CTA with more than kMaxOrder items keeps
  // the round order. sort_key packs (batch * head, item) into one 64-bit key.
  uint16_t* const order_sm = reinterpret_cast<uint16_t*>(smem + kOffOrder);
  const bool sorted_order = kCausal && n_mine <= kMaxOrder;
  auto sort_key = [&](int r) {
    const uint32_t it = static_cast<uint32_t>(item_of(r));
    return (static_cast<unsigned long long>(it % static_cast<uint32_t>(p.BH)) << 32) | it;
  };
  auto mine = [&](int k) { return item_of(sorted_order ? static_cast<int>(order_sm[k]) : k); };
  if (threadIdx.x == 0) {
    ATTN_STAMP(0);
    ATTN_STAMP_SM();
  }
  Ctl c;
  c.bar0 = base + kOffBar;
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kOffAbort);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  float* const alpha_sm = reinterpret_cast<float*>(smem + kOffAlpha);
  const uint32_t q_smem = base + kOffQ;
  const uint32_t kv_smem = base + kOffKV;

  auto load_q = [&](const Item& it, int q, uint64_t policy) {
    const uint32_t bar = c.bar(kBarQFull + q);
    const uint32_t dst = q_smem + q * kTileBytes;
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_4d_hint(dst, &tm_q, bar, 0, it.q0 + q * kBlock, it.hh, it.bb, policy);
    tma_load_4d_hint(dst + kSliceBytes, &tm_q, bar, 64, it.q0 + q * kBlock, it.hh, it.bb, policy);
  };
  // Global token T (K of the CTA's tile T/2 for even T, V for odd), local tile u/2 of item it.
  auto load_token = [&](const Item& it, int T, int u, uint64_t policy) {
    const uint32_t bar = c.bar(kBarKVFull + T % kStages);
    const uint32_t dst = kv_smem + (T % kStages) * kTileBytes;
    const CUtensorMap* map = (T & 1) ? &tm_v : &tm_k;
    const int row = (u >> 1) * kBlock;
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_4d_hint(dst, map, bar, 0, row, it.hh, it.bb, policy);
    tma_load_4d_hint(dst + kSliceBytes, map, bar, 64, row, it.hh, it.bb, policy);
  };

  // Set-up runs in a warp with no later role, so that no working warp ever runs diverged code.
  // With a sorted order it first finds the CTA's first item (the smallest key, a warp-wide
  // minimum), so that the first loads leave before the rest of the order is sorted.
  int r_first = 0;
  if (warp == kSetupWarp && sorted_order) {
    unsigned long long* const keys = reinterpret_cast<unsigned long long*>(smem + kOffStage);
    unsigned long long best = ~0ull;
    for (int r = lane; r < n_mine; r += 32) {
      keys[r] = sort_key(r);
      best = keys[r] < best ? keys[r] : best;
    }
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o < best ? o : best;
    }
    r_first = -1;
    for (int r = lane; r < n_mine; r += 32)
      if (keys[r] == best) r_first = r;
    for (int off = 16; off > 0; off >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, r_first, off);
      r_first = o > r_first ? o : r_first;
    }
    __syncwarp();
  }
  if (warp == kSetupWarp && lane == 0) {
    mbar_init(c.bar(kBarQFull + 0), 1);
    mbar_init(c.bar(kBarQFull + 1), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(c.bar(kBarKVFull + s), 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(c.bar(kBarSFull + q), 1);
      mbar_init(c.bar(kBarOSafe + q), 4);
      mbar_init(c.bar(kBarOFull + q), 1);
      mbar_init(c.bar(kBarStats + q), 4);
    }
    mbar_init(c.bar(kBarMmaDone + 0), 1);
    mbar_init(c.bar(kBarMmaDone + 1), 1);
    mbar_init(c.bar(kBarTurn + 0), 1);
    mbar_init(c.bar(kBarTurn + 1), 1);
    *c.abort_flag = 0u;
    reinterpret_cast<volatile int*>(smem + kOffFail)[0] = 0;
    reinterpret_cast<volatile int*>(smem + kOffFail)[1] = 0;
    reinterpret_cast<volatile int*>(smem + kOffSeen)[0] = 0;
    reinterpret_cast<volatile int*>(smem + kOffSeen)[1] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    const Item it = item_at(item_of(r_first));
    const uint64_t once = l2_policy_evict_first();
    load_q(it, 0, once);
    if (!ATTN_WITHHELD(p, 0)) load_token(it, 0, 0, l2_policy_evict_last());
    load_q(it, 1, once);
  }
  if (warp == kSetupWarp && sorted_order) {
    // Rank sort of the keys staged above in the O staging area (unused until the first epilogue).
    const unsigned long long* const keys = reinterpret_cast<const unsigned long long*>(smem + kOffStage);
    __syncwarp();
    for (int r = lane; r < n_mine; r += 32) {
      const unsigned long long kr = keys[r];
      int rank = 0;
      for (int r2 = 0; r2 < n_mine; ++r2) rank += keys[r2] < kr ? 1 : 0;
      order_sm[rank] = static_cast<uint16_t>(r);
    }
    __syncwarp();
  }
  if (warp == kTmemWarp) {
    tmem_alloc(base + kOffTmemSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) ATTN_STAMP(1);
  volatile int* const issuer_stopped = reinterpret_cast<volatile int*>(smem + kOffFail);
  // s_seen[q]: how many S_q tiles the softmax warps have seen complete (the CTA's global tile
  // count). S_q(g) complete means QK_q(g) and every earlier MMA of Q tile q have finished, and
  // the MMAs of Q tile 0 run ahead of those of Q tile 1 in the same tensor pipe.
  volatile int* const s_seen = reinterpret_cast<volatile int*>(smem + kOffSeen);

  if (warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
  }
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      // Every wait is on the softmax warps' S-seen counts, which only grow. (A parity wait on the
      // S barriers themselves could run two phases ahead of them at an item boundary, or find
      // them two phases on, and take a wrong phase for the one it needs.)
      const uint32_t code0 = 0xA77E0000u | (kRoleLoad << 8) | static_cast<uint32_t>(kSeenCode);
      bool ok = true;
      int issued = 1;           // global token 0 (the first item's K0) was loaded at set-up
      int gbase = 0;            // global index of the item's first K/V tile
      int q_loads[2] = {1, 1};  // Q tile loads so far (the phases of the Q barriers)
      for (int k = 0; k < n_mine && ok; ++k) {
        const Item it = item_at(mine(k));
        for (int u = 0; u < 2 * it.n; ++u) {
          const int T = 2 * gbase + u;
          if (T == 0) continue;
          if (k > 0 && u == 0) {
            // Q_0 of this item replaces the previous item's once QK_0 of its last tile is done.
            if (!wait_count(c, s_seen + 0, gbase, code0)) { ok = false; break; }
            load_q(it, 0, once);
            ++q_loads[0];
          }
          if (T >= kStages) {
            // The slot's previous token: K of tile g is free once QK_1(g) is done, V of tile g
            // once QK_1(g + 1) is (its commit covers PV_1(g)); Q tile 0's MMAs run first.
            const int prev = T - kStages;
            if (!wait_count(c, s_seen + 1, prev / 2 + 1 + (prev & 1), code0 + 1)) { ok = false; break; }
          }
          if (!ATTN_WITHHELD(p, T)) load_token(it, T, u, keep);
          issued = T + 1;
          if (k > 0 && u == 0) {
            if (!wait_count(c, s_seen + 1, gbase, code0 + 1)) { ok = false; break; }
            load_q(it, 1, once);
            ++q_loads[1];
          }
        }
        gbase += it.n;
      }
      if (!ok) {
        // Drain: the last load of each Q tile and of the ring slots still owed.
        for (int q = 0; q < 2; ++q)
          wait_slow(c, kBarQFull + q, static_cast<uint32_t>((q_loads[q] - 1) & 1), kRoleLoad, false, kDrainLimitNs);
        for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
          if (!ATTN_WITHHELD(p, t))
            wait_slow(c, kBarKVFull + t % kStages, (t / kStages) & 1, kRoleLoad, false, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == kIssueWarp0 || warp == kIssueWarp1) {
    // ------------------------------------------------------------------ MMA issue (Q tile q)
    const int q = warp == kIssueWarp1 ? 1 : 0;
    const uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t kIdescPV = idesc_bf16_f32(128, 128, 0, 1);
    constexpr uint32_t kTileUnits = kTileBytes >> 4;
    const uint32_t tSq = tmem + q * 128u, tOq = tmem + 256u + q * 128u;
    const uint64_t dq = smem_desc_sw128(q_smem + q * kTileBytes, 16, 1024);
    const uint64_t dk = smem_desc_sw128(kv_smem, 16, 1024);
    const uint64_t dv = smem_desc_sw128(kv_smem, kSliceBytes, 1024);
    auto issue_qk = [&](uint32_t k_slot, bool hand_over) {
      const uint64_t b0 = dk + k_slot * kTileUnits;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = ((kk >> 2) * kSliceBytes + (kk & 3) * 32) >> 4;
        mma_bf16_ss(tSq, dq + off, b0 + off, kIdescQK, kk > 0 ? 1u : 0u);
        if (hand_over && kk == 7) {
          tc_fence_before();
          mbar_arrive(c.bar(kBarTurn + (q ^ 1)));
        }
      }
    };
    auto issue_pv = [&](uint32_t v_slot, int k0, int k1, bool first) {
      const uint64_t b0 = dv + v_slot * kTileUnits;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (kk >= k0 && kk < k1)
          mma_bf16_ts(tOq, tSq + kk * 8, b0 + kk * (2048 >> 4), kIdescPV, (first && kk == 0) ? 0u : 1u);
    };
    auto token_bar = [&](int t) { return kBarKVFull + t % kStages; };
    auto token_par = [&](int t) { return static_cast<uint32_t>((t / kStages) & 1); };
    bool ok = true;
    if (lane == 0) {
      ok = wait_bar(c, kBarQFull + q, 0, kRoleMma) && wait_bar(c, token_bar(0), 0, kRoleMma) &&
           (q == 0 || wait_bar(c, kBarTurn + 1, 0, kRoleMma));
      if (ok) {
        tc_fence_after();
        issue_qk(0, false);
        mma_commit(c.bar(kBarSFull + q));
        tc_fence_before();
        mbar_arrive(c.bar(kBarTurn + (q ^ 1)));
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    // One flat loop over the CTA's stream of K/V tiles: gt counts tiles across items, i is the
    // tile within the current item, n its tile count.
    int k = 0;
    int n = kCausal ? item_at(mine(0)).n : p.n_kv;
    bool next_item = 1 < n_mine;
    for (int gt = 0, i = 0; ok; ++gt) {
      const int tv = 2 * gt + 1, tk = 2 * gt + 2;
      const bool more = i + 1 < n;
      auto part = [&](auto pc) {
        constexpr int pi = decltype(pc)::value;
        constexpr int c0 = kPCut[pi], c1 = kPCut[pi + 1];
        named_bar_sync(kBarP + 2 * pi + q, 160);
        if (ok && lane == 0) {
          tc_fence_after();
          if constexpr (pi == 0) {
            const uint32_t turn_par = static_cast<uint32_t>((q == 0 ? gt : gt + 1) & 1);
            const uint32_t rdy = mbar_probe4(c.bar(token_bar(tv)), token_par(tv),
                                             c.bar(kBarOSafe + q), static_cast<uint32_t>((gt - 1) & 1),
                                             c.bar(kBarTurn + q), turn_par,
                                             c.bar(kBarTurn + q), turn_par);
            ok = ((rdy & 1u) || wait_bar(c, token_bar(tv), token_par(tv), kRoleMma)) &&
                 (gt == 0 || (rdy & 2u) || wait_bar(c, kBarOSafe + q, (gt - 1) & 1, kRoleMma)) &&
                 ((rdy & 4u) || wait_bar(c, kBarTurn + q, turn_par, kRoleMma));
          }
          if constexpr (pi == kPParts - 1) ok = ok && (!more || wait_bar(c, token_bar(tk), token_par(tk), kRoleMma));
          if (ok) {
            tc_fence_after();
            issue_pv(static_cast<uint32_t>(tv % kStages), c0 / 8, c1 / 8, pi == 0 && i == 0);
            ATTN_STAMP_IF(q == 0 && k == 1 && pi == 0 && i == 0, 15);
            if constexpr (pi == kPParts - 1) {
              if (more) {
                issue_qk(static_cast<uint32_t>(tk % kStages), true);
                mma_commit(c.bar(kBarSFull + q));
              } else {
                mma_commit(c.bar(kBarOFull + q));
                if (next_item) {
                  ok = wait_bar(c, token_bar(tk), token_par(tk), kRoleMma) &&
                       wait_bar(c, kBarQFull + q, static_cast<uint32_t>((k + 1) & 1), kRoleMma);
                  if (ok) {
                    tc_fence_after();
                    issue_qk(static_cast<uint32_t>(tk % kStages), true);
                    mma_commit(c.bar(kBarSFull + q));
                    ATTN_STAMP_IF(q == 0 && k == 0, 14);
                  }
                } else if (q == 0) {
                  tc_fence_before();
                  mbar_arrive(c.bar(kBarTurn + 1));
                }
              }
            }
          }
        }
      };
      static_for<kPParts>(part);
      // Lanes 1-31 only wait at the named barriers; they need lane 0's result for the loop test.
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (more) {
        ++i;
      } else {
        ++k;
        if (!next_item) break;
        i = 0;
        n = kCausal ? item_at(mine(k)).n : p.n_kv;
        next_item = k + 1 < n_mine;
      }
    }
    if (!ok && lane == 0) {
      // No further QK for this tile: the softmax warps waiting for one may leave.
      issuer_stopped[q] = 1;
      __threadfence_block();
    }
    if (lane == 0) {
      const bool fin = ok && wait_bar(c, kBarOFull + q, static_cast<uint32_t>((k - 1) & 1), kRoleMma);
      if (!fin) {
        mma_commit(c.bar(kBarMmaDone + q));
        wait_slow(c, kBarMmaDone + q, 0, kRoleMma, false, kDrainLimitNs);
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------------ softmax (Q tile q)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;");
    const int q = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t tS = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + q * 128u;
    const float sl2 = p.scale_log2;
    const int rem = p.S - (p.n_kv - 1) * kBlock;
    const uint32_t stage = base + kOffStage + (q * 4 + (warp & 3)) * kStageWarpBytes;
    bool ok = true;
    int gbase = 0, k = 0;
    for (; k < n_mine && ok; ++k) {
      const Item it = item_at(mine(k));
      const bool next_item = k + 1 < n_mine;
      float m_kept = -INFINITY;
      float l = 0.f;
      float lf = 0.f;
      for (int i = 0; i < it.n; ++i) {
        const int gt = gbase + i;
        if (!wait_s_full(c, kBarSFull + q, gt & 1, issuer_stopped + q)) {
          ok = false;  // no QK_q(gt) is coming: leave without arriving at its barriers
          break;
        }
        if ((warp & 3) == 0 && lane == 0) st_release_shared(s_seen + q, gt + 1);
        ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 0 && i == it.n - 1, 8);
        ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 1 && i == 0, 12);
        if (gt == 0 && warp == 0 && lane == 0) ATTN_STAMP(2);
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld32_x128_sync(tS, sr);
        float s[128];
#pragma unroll
        for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(sr[j]);
        if (i == p.n_kv - 1 && rem < kBlock) {
#pragma unroll
          for (int j = 0; j < 128; ++j) s[j] = (j < rem) ? s[j] : -INFINITY;
        }
        if (kCausal && i >= 2 * it.qp + q) {
          const int lim = it.q0 + q * kBlock + row - i * kBlock;
#pragma unroll
          for (int j = 0; j < 128; ++j) s[j] = (j <= lim) ? s[j] : -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) mx[j] = fmaxf(s[2 * j], s[2 * j + 1]);
#pragma unroll
        for (int j = 8; j < 128; j += 8) {
          mx[0] = max3(mx[0], s[j + 0], s[j + 1]);
          mx[1] = max3(mx[1], s[j + 2], s[j + 3]);
          mx[2] = max3(mx[2], s[j + 4], s[j + 5]);
          mx[3] = max3(mx[3], s[j + 6], s[j + 7]);
        }
        const float tile_max = max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sl2;
        if (i == 0) {
          m_kept = tile_max;
        } else {
          float alpha = 1.0f;
          if (kThr == 0 ? (tile_max > m_kept) : (tile_max - m_kept >= static_cast<float>(kThr))) {
            alpha = ex2_ftz(m_kept - tile_max);
            if constexpr (kThr == 8) l *= alpha;
            lf *= alpha;
            m_kept = tile_max;
          }
          alpha_sm[q * kBlock + row] = alpha;
          warp_arrive(c, kBarStats + q, lane);
        }
        const float neg_m = -m_kept;
        float lb0 = 0.f, lb1 = 0.f, lb2 = 0.f, lb3 = 0.f;
        float lf0 = 0.f, lf1 = 0.f, lf2 = 0.f, lf3 = 0.f;
        uint32_t pk[64];
        auto pair = [&](int j) {
          float x0, x1;
          fma2(x0, x1, s[2 * j], s[2 * j + 1], sl2, sl2, neg_m, neg_m);
          const float p0 = ex2_ftz(x0);
          const float p1 = ex2_ftz(x1);
          pk[j] = pack_bf16x2(p0, p1);
          if (j & 1) {
            add2(lf2, lf3, lf2, lf3, p0, p1);
          } else {
            add2(lf0, lf1, lf0, lf1, p0, p1);
          }
          if constexpr (kThr == 8) {
            float b0, b1;
            bf16x2_to_f32x2(pk[j], b0, b1);
            if (j & 1) add2(lb2, lb3, lb2, lb3, b0, b1);
            else add2(lb0, lb1, lb0, lb1, b0, b1);
          }
        };
        auto part = [&](auto pc) {
          constexpr int pi = decltype(pc)::value;
          constexpr int c0 = kPCut[pi], c1 = kPCut[pi + 1];
#pragma unroll
          for (int j = c0; j < c1; ++j) pair(j);
          tmem_st_cols<c0, c1>(tS, pk);
          tmem_wait_st();
          tc_fence_before();
          named_bar_arrive(kBarP + 2 * pi + q, 160);
          ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 0 && pi == kPParts - 1 && i == it.n - 1, 9);
          ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 1 && pi == 0 && i == 0, 13);
        };
        static_for<kPParts>(part);
        lf += (lf0 + lf1) + (lf2 + lf3);
        if constexpr (kThr == 8) l += (lb0 + lb1) + (lb2 + lb3);
        else l = lf;
      }
      if (!ok) break;
      const bool fin = wait_bar_warp(c, kBarOFull + q, static_cast<uint32_t>(k & 1), kRoleSoftmax);
      if (k == 0 && (warp & 3) == 0 && lane == 0) ATTN_STAMP(3 + q);
      if (!fin) {
        ok = false;
        break;
      }
      // epilogue: O / l -> BF16 -> this warp's 4 KB staging (32 rows x 64 columns, SW128) ->
      // TMA store, twice (columns 0-63, 64-127). O_q is released to the next item's first PV as
      // soon as it has been read out of tensor memory.
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const uint32_t tO = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 256u + q * 128u;
      uint32_t o[128];
      tmem_ld32_x128_sync(tO, o);
      if (next_item) {
        tc_fence_before();
        warp_arrive(c, kBarOSafe + q, lane);  // O_q drained
      }
      ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 0, 10);
      const int r0 = it.q0 + q * kBlock + (warp & 3) * 32;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (half == 1 || k > 0) {
          // the previous store out of this staging has been read
          if (lane == 0) tma_store_wait_read_all();
          __syncwarp();
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int cc = half * 8 + ch;
          uint32_t w4[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            w4[t] = pack_bf16x2(__uint_as_float(o[8 * cc + 2 * t]) * inv_l,
                                __uint_as_float(o[8 * cc + 2 * t + 1]) * inv_l);
          const uint32_t addr = stage + lane * 128 + (static_cast<uint32_t>(ch ^ (lane & 7)) << 4);
          st_shared_v4(addr, w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && r0 < p.S) {
          tma_store_4d(&tm_o, stage, half * 64, r0, it.hh, it.bb);
          tma_store_commit();
        }
        __syncwarp();
      }
      const int grow = it.q0 + q * kBlock + row;
      if (p.lse != nullptr && grow < p.S)
        p.lse[static_cast<size_t>(it.bh) * p.S + grow] = (m_kept + log2f(lf)) * 0.69314718055994531f;
      ATTN_STAMP_IF(warp == 0 && lane == 0 && k == 0, 11);
      gbase += it.n;
    }
    if (lane == 0) tma_store_wait_read_all();
    __syncwarp();
  } else if (warp < 12) {
    // ------------------------------------------------------------------ correction
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;");
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_field = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO[2] = {tmem + lane_field + 256u, tmem + lane_field + 384u};
    bool ok = true;
    int sbase = 0;  // stats phases before this item
    for (int r = 0; r < n_mine && ok; ++r) {
      const Item it = item_at(mine(r));
      for (int i = 1; i < it.n && ok; ++i) {
        for (int q = 0; q < 2; ++q) {
          {
            if (!wait_bar_warp(c, kBarStats + q, static_cast<uint32_t>((sbase + i - 1) & 1), kRoleCorrection)) {
              ok = false;
              break;
            }
            const float alpha = alpha_sm[q * kBlock + row];
            if (__any_sync(0xffffffffu, alpha != 1.0f)) {
              tc_fence_after();
#pragma unroll 1
              for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32_x32_sync(tO[q] + cc * 32, o);
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                  float a0, a1;
                  fma2(a0, a1, __uint_as_float(o[j]), __uint_as_float(o[j + 1]), alpha, alpha, 0.f, 0.f);
                  o[j] = __float_as_uint(a0);
                  o[j + 1] = __float_as_uint(a1);
                }
                tmem_st32_x32(tO[q] + cc * 32, o);
              }
              tmem_wait_st();
            }
            tc_fence_before();
          }
          warp_arrive(c, kBarOSafe + q, lane);
        }
      }
      sbase += it.n - 1;
    }
  }

  if (threadIdx.x == 0) ATTN_STAMP(5);
  tc_fence_before();
  __syncthreads();
  if (warp == kTmemWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) ATTN_STAMP(7);
}

}  // namespace gb300

// ==========================================================================================
// Host side
// ==========================================================================================
namespace gb300 {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, -1 unsupported/failed
int g_dev_sms[kMaxDevices];                 // SM count, set before the device is marked ready
std::mutex g_dev_mutex;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Checks the device once (compute capability 10.3) and sets the kernel's shared-memory limit.
int prepare_device(int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  *dev_out = dev;
  if (dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 1) return ATTN_OK;
  if (st == -1) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st != 0) return st == 1 ? ATTN_OK : ATTN_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3) {
    cudaGetLastError();
    g_dev_state[dev].store(-1, std::memory_order_release);
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  auto smem_attr = [](const void* fn) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) == cudaSuccess;
  };
  if (!smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<0, false>)) ||
      !smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<1, false>)) ||
      !smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<8, false>)) ||
      !smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<0, true>)) ||
      !smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<1, true>)) ||
      !smem_attr(reinterpret_cast<const void*>(attn_fwd_kernel<8, true>))) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  g_dev_sms[dev] = sms;
  g_dev_state[dev].store(1, std::memory_order_release);
  return ATTN_OK;
}

// A BF16 [B, H, S, D] tensor with element strides (sb, sh, ss) and unit stride along D, as a
// 4-D tensor map {D, S, H, B}; 64 x box_rows boxes (128 for loads, 32 for the per-warp
// output stores), 128-byte swizzle, zero fill past S.
bool encode_4d(CUtensorMap* map, const void* ptr, int B, int H, int S, const long long (&st)[3],
               int box_rows = kBlock) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                                 static_cast<cuuint64_t>(st[0]) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bytes from the first to one past the last element a strided [B, H, S, 128] tensor touches.
size_t span_bytes(int B, int H, int S, const long long (&st)[3]) {
  return static_cast<size_t>((static_cast<long long>(B - 1) * st[0] + static_cast<long long>(H - 1) * st[1] +
                              static_cast<long long>(S - 1) * st[2] + kHeadDim) *
                             2);
}

// Element strides that map distinct (b, h, s, d) to distinct addresses: sorted by size,
// each stride covers the extent of the next smaller one (a row of 128 for the smallest).
bool injective(int B, int H, int S, const long long (&st)[3]) {
  long long v[3][2] = {{st[0], B}, {st[1], H}, {st[2], S}};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (v[j][0] < v[i][0]) {
        std::swap(v[i][0], v[j][0]);
        std::swap(v[i][1], v[j][1]);
      }
  long long need = kHeadDim;
  for (int i = 0; i < 3; ++i) {
    if (v[i][1] > 1) {
      if (v[i][0] < need) return false;
      need = v[i][0] * v[i][1];
    }
  }
  return true;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace gb300

extern "C" {

static int attn_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                       int S, int D, float scale, const long long* qs, const long long* ks,
                       const long long* vs, const long long* os, int rebase_threshold_log2,
                       int causal, int withhold, int check_only, void* stream) {
  using namespace gb300;
  if (rebase_threshold_log2 != 0 && rebase_threshold_log2 != 1 && rebase_threshold_log2 != 8)
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (D != kHeadDim) return ATTN_ERR_UNSUPPORTED_DIM;
  if (!q || !k || !v || !o || !qs || !ks || !vs || !os) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || S <= 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_qp = (static_cast<long long>(S) + 2 * kBlock - 1) / (2 * kBlock);
  if (BH > (1ll << 31) - 1 || BH * n_qp > (1ll << 31) - 1) return ATTN_ERR_INVALID_ARG;
  const long long n_kv = (static_cast<long long>(S) + kBlock - 1) / kBlock;
  if (withhold < -1 || withhold >= 2 * n_kv) return ATTN_ERR_INVALID_ARG;
  long long st[4][3];
  const long long* in[4] = {qs, ks, vs, os};
  for (int t = 0; t < 4; ++t) {
    for (int j = 0; j < 3; ++j) {
      st[t][j] = in[t][j];
      // TMA: strides in bytes are positive multiples of 16 below 2^40.
      if (st[t][j] <= 0 || st[t][j] >= (1ll << 39)) return ATTN_ERR_INVALID_ARG;
      if (st[t][j] % 8 != 0) return ATTN_ERR_MISALIGNED;
    }
  }
  if (!injective(B, H, S, st[3])) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_MISALIGNED;
  const size_t qb = span_bytes(B, H, S, st[0]), kb = span_bytes(B, H, S, st[1]);
  const size_t vb = span_bytes(B, H, S, st[2]), ob = span_bytes(B, H, S, st[3]);
  const size_t lse_bytes = static_cast<size_t>(BH) * S * 4;
  if (overlaps(o, ob, q, qb) || overlaps(o, ob, k, kb) || overlaps(o, ob, v, vb)) return ATTN_ERR_INVALID_ARG;
  if (lse && (overlaps(lse, lse_bytes, q, qb) || overlaps(lse, lse_bytes, k, kb) ||
              overlaps(lse, lse_bytes, v, vb) || overlaps(lse, lse_bytes, o, ob)))
    return ATTN_ERR_INVALID_ARG;

  if (check_only == 2) return ATTN_OK;  // arguments only, no CUDA call

  int dev = -1;
  const int status = prepare_device(&dev);
  if (status != ATTN_OK) return status;
  if (!get_encoder()) return ATTN_ERR_LAUNCH;
  if (check_only) return ATTN_OK;

  CUtensorMap tq, tk, tv, to;
  if (!encode_4d(&tq, q, B, H, S, st[0]) || !encode_4d(&tk, k, B, H, S, st[1]) ||
      !encode_4d(&tv, v, B, H, S, st[2]) || !encode_4d(&to, o, B, H, S, st[3], 32))
    return ATTN_ERR_LAUNCH;

  Params prm;
  prm.lse = lse;
  prm.S = S;
  prm.H = H;
  prm.n_kv = static_cast<int>(n_kv);
  prm.n_qp = static_cast<int>(n_qp);
  prm.BH = static_cast<int>(BH);
  prm.num_items = static_cast<int>(BH * n_qp);
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
#ifdef ATTN_TEST_HOOKS
  prm.withhold = withhold;
#endif

  // One CTA per SM (the kernel holds all of an SM's tensor memory); each CTA walks its items.
  const long long items = BH * n_qp;
  const int sms = g_dev_sms[dev];
  const dim3 grid(static_cast<unsigned>(items > sms ? sms : items));
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  auto launch = [&](auto kernel) { kernel<<<grid, kThreads, kSmemBytes, st_>>>(tq, tk, tv, to, prm); };
  if (rebase_threshold_log2 == 8) {
    if (causal) launch(attn_fwd_kernel<8, true>);
    else launch(attn_fwd_kernel<8, false>);
  } else if (rebase_threshold_log2 == 1) {
    if (causal) launch(attn_fwd_kernel<1, true>);
    else launch(attn_fwd_kernel<1, false>);
  } else {
    if (causal) launch(attn_fwd_kernel<0, true>);
    else launch(attn_fwd_kernel<0, false>);
  }
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int S, int D, float scale, int rebase_threshold_log2, void* stream) {
  // Contiguous [B, H, S, D]: element strides (H*S*D, S*D, D).
  const long long st[3] = {static_cast<long long>(H) * S * D, static_cast<long long>(S) * D, D};
  return attn_launch(q, k, v, o, lse, B, H, S, D, scale, st, st, st, st, rebase_threshold_log2, 0, -1, 0,
                     stream);
}

int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int S, int D, float scale, const long long* q_strides, const long long* k_strides,
                     const long long* v_strides, const long long* o_strides, int rebase_threshold_log2,
                     int causal, void* stream) {
  return attn_launch(q, k, v, o, lse, B, H, S, D, scale, q_strides, k_strides, v_strides, o_strides,
                     rebase_threshold_log2, causal, -1, 0, stream);
}

int attn_fwd_causal(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int S, int D, float scale, void* stream) {
  const long long st[3] = {static_cast<long long>(H) * S * D, static_cast<long long>(S) * D, D};
  return attn_launch(q, k, v, o, lse, B, H, S, D, scale, st, st, st, st, gb300::kDefaultRebase, 1, -1, 0, stream);
}

#ifdef ATTN_TEST_HOOKS
int attn_fwd_withhold(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int S, int D, float scale, int token, void* stream) {
  if (token < 0) return ATTN_ERR_INVALID_ARG;
  const long long st[3] = {static_cast<long long>(H) * S * D, static_cast<long long>(S) * D, D};
  return attn_launch(q, k, v, o, lse, B, H, S, D, scale, st, st, st, st, gb300::kDefaultRebase, 0, token, 0, stream);
}
#endif

int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, void* q_d,
                  void* k_d, void* v_d, void* o_d, float* lse_d, int B, int H, int S, int D, float scale,
                  int causal, void* stream) {
  if (!q_h || !k_h || !v_h || !o_h) return ATTN_ERR_INVALID_ARG;
  if ((lse_h == nullptr) != (lse_d == nullptr)) return ATTN_ERR_INVALID_ARG;
  const long long st[3] = {static_cast<long long>(H) * S * D, static_cast<long long>(S) * D, D};
  // Everything the kernel launch would reject is rejected before any copy is enqueued.
  int r = attn_launch(q_d, k_d, v_d, o_d, lse_d, B, H, S, D, scale, st, st, st, st, gb300::kDefaultRebase, causal, -1, 2, stream);
  if (r != ATTN_OK) return r;
  const size_t bytes = static_cast<size_t>(B) * H * S * D * 2;
  const size_t lse_bytes = static_cast<size_t>(B) * H * S * 4;
  // q_d, k_d and v_d are copy destinations here (the kernel alone may read aliased inputs):
  // one copy would overwrite another's data.
  if (gb300::overlaps(q_d, bytes, k_d, bytes) || gb300::overlaps(q_d, bytes, v_d, bytes) ||
      gb300::overlaps(k_d, bytes, v_d, bytes))
    return ATTN_ERR_INVALID_ARG;
  r = attn_launch(q_d, k_d, v_d, o_d, lse_d, B, H, S, D, scale, st, st, st, st, gb300::kDefaultRebase, causal, -1, 1, stream);
  if (r != ATTN_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(q_d, q_h, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(k_d, k_h, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(v_d, v_h, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  r = attn_launch(q_d, k_d, v_d, o_d, lse_d, B, H, S, D, scale, st, st, st, st, gb300::kDefaultRebase, causal, -1, 0, stream);
  if (r != ATTN_OK) return r;
  if (cudaMemcpyAsync(o_h, o_d, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (lse_h && cudaMemcpyAsync(lse_h, lse_d, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int S, int D, float scale, void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, S, D, scale, gb300::kDefaultRebase, stream);
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED_DIM: return "unsupported head dimension (D must be 128)";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (q/k/v/o need 16 bytes, lse 4)";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "no CUDA device, or the device is not sm_103";
    case ATTN_ERR_LAUNCH: return "tensor-map encoding or kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

int attn_device_status(unsigned int* word, int reset) {
  if (!word) return ATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  unsigned int w = 0;
  if (cudaMemcpyFromSymbol(&w, gb300::g_attn_status, sizeof(w)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  if (reset && w != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(gb300::g_attn_status, &zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
  }
  *word = w;
  return ATTN_OK;
}

int attn_version(void) { return (1 << 16) | 0; }

#ifdef ATTN_TRACE
int attn_trace_read(unsigned long long* out, int max_ctas) {
  if (!out || max_ctas <= 0) return ATTN_ERR_INVALID_ARG;
  const int nct = max_ctas < ATTN_TRACE_CTAS ? max_ctas : ATTN_TRACE_CTAS;
  if (cudaMemcpyFromSymbol(out, gb300::g_attn_trace, static_cast<size_t>(nct) * gb300::kTraceWords * sizeof(unsigned long long)) !=
      cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int attn_trace_clear(void) {
  static unsigned long long zero[ATTN_TRACE_CTAS * gb300::kTraceWords];
  if (cudaMemcpyToSymbol(gb300::g_attn_trace, zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}
#endif

}  // extern "C"
