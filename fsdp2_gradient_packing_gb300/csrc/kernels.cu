// sm_103a kernels and the launching entry points of the C ABI.
//
// The four packing operations (reduce-scatter copy-in, all-gather copy-in,
// all-gather copy-out, reduce-scatter copy-out) are all "walk a table of
// contiguous runs and copy each one with a cast": dst[k] = k < n_copy ?
// cast(src[k]) : +0 for k < n_total.  The host planner (plan.cpp) emits the
// runs once per layout, cut into work items of at most kStageBytes of source;
// one launch per call walks them (walk_kernel), or, for the *_batched calls,
// one launch walks the tables of up to 64 layouts.  Every launch but the
// allocation-free pack's uses programmatic dependent launch: it may be
// scheduled while the previous kernel on the stream drains, and waits for it
// before touching memory; meanwhile it prefetches the sources of its first
// items into L2, a hint that reads nothing into the CTA.  A separate
// elementwise kernel (sum_kernel, in reduce.cu) serves the emulated
// reduce-scatter.
//
// The work is bound by HBM bandwidth, so the kernel is a warp-specialised
// pipeline built to keep many bytes in flight per SM with few registers and
// to write only full, aligned 16-byte vectors:
//   * warp 0, lane 0 is the producer (in short single launches the warp's
//     lanes first resolve the CTA's first items -- descriptor and source /
//     destination pointers -- in parallel, one per lane, and the lanes
//     stage the ring's first fill together).  For each item of its CTA the
//     producer copies the item's source bytes, widened to whole aligned
//     16-byte blocks, into one stage of a shared-memory ring with one TMA
//     bulk copy (cp.async.bulk), completion counted on that stage's "full"
//     mbarrier;
//   * warps 1..8 are consumers.  For each item they wait on the stage, then
//     write the destination as 16-byte vectors: each lane reads the source
//     bytes of one vector from shared memory at whatever byte phase they have
//     (word loads plus a funnel shift), converts them and stores one aligned
//     16-byte vector, so every warp store covers 512 contiguous bytes.  Vectors
//     made only of padding are stored as zeros without reading anything.
//     The destination's head before its first 16-byte boundary, its tail, and
//     the one vector where valid data meets padding are written element by
//     element, also from the stage: consumers never read global memory;
//   * consumers release the stage on its "empty" mbarrier; the producer
//     reuses it kStages items later.
// FP32 -> BF16 rounding in walk_kernel is done on the bits (round to nearest,
// ties to even), so results do not depend on the device's FP modes; the
// vector path of sum_kernel adds BF16 pairs with the hardware's BF16
// addition (round to nearest even), which gives the same bits.
//
// Every mbarrier wait is bounded (a limit in nanoseconds of %globaltimer).  A
// wait that gives up sets a bit in the layout's device status word and the
// thread leaves; the producer first waits (again bounded) for the bulk copies
// it issued, so no copy is in flight when its CTA exits.  fsdp_sync_status()
// reads and clears that word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "bf16_bits.h"
#include "layout.h"

namespace fsdp {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kStages = 4;
// Each stage holds the item's staged source -- its source bytes widened to
// whole aligned 16-byte blocks, at most kStageBytes + 16 bytes, plus slack
// for the funnel read of the last vector, which may touch one word past them
// -- and after it a 64-byte header (the item, see StageHeader).  Stages start
// on 128-byte boundaries, where the bulk copies write them.
constexpr int kStagedMax = (int)kStageBytes + 16;
constexpr int kStageDataBytes = (int)kStageBytes + 32;
constexpr int kHeaderBytes = 64;
constexpr int kStageStride = (kStageDataBytes + kHeaderBytes + 127) / 128 * 128;
static_assert(kStageDataBytes % 16 == 0, "stage header must stay 16-byte aligned");
// After the stages: their "full" and "empty" barriers, then the resolved
// headers of a CTA's first kPrefetch items (StageHeader, 32 bytes each; see
// the producer prologue).  The prologue runs in launches of at most
// kPrologueMaxRounds items per CTA.
constexpr int kPrefetch = 32;
constexpr int64_t kPrologueMaxRounds = 64;
// Items per CTA whose staged source is prefetched into L2 before the
// dependent-launch wait: the ones that fill the ring first, in a CTA that has
// more fixed-order items than that to follow.  A CTA whose whole work fits the
// ring prefetches its first item only.  Without the parallel prologue the
// producer looks them up one after another, which pays off only in launches
// of at least kSeqPrefetchMinRounds items per CTA; shorter ones look up (and
// prefetch) item 0 alone.
constexpr int kL2PrefetchItems = kStages;
constexpr int64_t kSeqPrefetchMinRounds = 16;
constexpr int kMaxBatch = 64;  // layouts in one batched launch
constexpr int kBarrierBytes = 2 * kStages * 8;
constexpr int kPrefetchOffset = kStages * kStageStride + kBarrierBytes;
constexpr int kSmemBytes = kPrefetchOffset + kPrefetch * 32;
static_assert(kPrefetchOffset % 16 == 0, "shared tables must stay 16-byte aligned");
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// Status bits written by a kernel whose bounded wait gave up.
constexpr uint32_t kStatusConsumerWait = 1u;
constexpr uint32_t kStatusProducerWait = 2u;
constexpr uint32_t kStatusDrainWait = 4u;
constexpr uint32_t kStatusBadItem = 8u;

// Test hook: the producer of CTA 0 does not arm its first stage, so that
// stage's consumers time out (no fault, no hang: every wait is bounded).
constexpr int32_t kFaultSkipFirstStage = 1;

// How a launch hands out its n work items to its G CTAs.  CTA b first takes
// items b + m*G for m < fixed_rounds, in that fixed order.  The rest, items
// [fixed_rounds*G, n), go to whichever CTA asks first, through a work-sharing
// word in device memory (one per layout and operation); with word == nullptr
// they follow the fixed order too.  See sched_join for the word's protocol.
struct Sched {
  unsigned long long *word;
  int64_t fixed_rounds;
  uint32_t tag;   // this launch's owner tag: nonzero, 24 bits
  int32_t flags;  // kSchedMixed
};
// Test hook: CTAs with an odd index act as if another launch held the word,
// so one launch mixes CTAs that share the word with CTAs in the fixed order.
constexpr int32_t kSchedMixed = 1;

// Per-call pointers travel by value in the parameter block: `slot` is read
// with a run-time index, which __grid_constant__ allows without a local copy.
// fetch(i) returns work item i and the slot base its slot numbers are
// relative to; `cursor` carries the layout of the CTA's previous item.
template <int NSLOT>
struct LaunchArgs {
  // The producer warp's lanes resolve the CTA's first items in parallel
  // (see the producer prologue in walk_kernel).
  static constexpr bool kParallelPrologue = true;
  const WorkItem *items;
  int64_t n_items;
  uint32_t *status;
  uint64_t wait_limit_ns;
  int32_t fault;
  int32_t reserved;
  Sched sched;
  const void *slot[NSLOT];

  __device__ __forceinline__ WorkItem fetch(int64_t i, int32_t *base, int *) const {
    *base = 0;
    return items[i];
  }
};

// Several layouts in one launch: the items of layout g are global items
// [start[g], start[g+1]); their slots are numbered from slot_base[g].
template <int NSLOT>
struct BatchArgs {
  // A batched launch resolves its items one at a time on the producer lane.
  // Resolved by a warp's lanes at once, the lookups would index the
  // per-layout arrays and the slots of the parameter block with a different
  // index in every lane, which the constant cache serves one address after
  // another: measured slower than the sequential producer.
  static constexpr bool kParallelPrologue = false;
  int64_t n_items;
  uint32_t *status;
  uint64_t wait_limit_ns;
  int32_t fault;
  int32_t n_groups;
  Sched sched;
  const WorkItem *items[kMaxBatch];
  int64_t start[kMaxBatch + 1];
  int32_t slot_base[kMaxBatch];
  const void *slot[NSLOT];

  // The last group that starts at or before i, found by walking forward
  // from the CTA's previous one: a CTA's item indices grow (except after the
  // rare retake of the work-sharing word, which restarts the walk), so the
  // walk costs about one step per layout instead of a chain of dependent
  // parameter loads per item.
  __device__ __forceinline__ WorkItem fetch(int64_t i, int32_t *base, int *cursor) const {
    int g = *cursor;
    if (start[g] > i) g = 0;
    while (g + 1 < n_groups && start[g + 1] <= i) ++g;
    *cursor = g;
    *base = slot_base[g];
    return items[g][i - start[g]];
  }
};

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk copy, timer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete, for at most limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Programmatic dependent launch.  Every launch allows the next kernel on the
// stream to be scheduled early (launch_dependents), and waits for the
// previous kernel on the stream to finish and publish its memory
// (griddepcontrol.wait) before touching any input or output.  Only the work
// table and the parameter block are read before the wait: a layout's table
// never changes after planning, and the allocation-free pack, whose table is
// rewritten before each of its launches, launches without programmatic
// serialization (see noalloc_launch).
__device__ __forceinline__ void wait_for_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One TMA bulk copy global -> shared, completion counted on `bar` in bytes.
// Both addresses are 16-byte aligned and `bytes` is a multiple of 16.  The
// source is read exactly once, so its lines are marked first to be evicted
// from L2, which leaves L2 to the destination's write-combining.
__device__ __forceinline__ void bulk_copy_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                              uint64_t *bar) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// One aligned 16-byte store of the destination.
__device__ __forceinline__ void store_vec(uint4 *d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
  *d = make_uint4(a0, a1, a2, a3);
}

// ---------------------------------------------------------------------------
// Element types of each conversion kind (the conversions themselves, on raw
// bits, are in bf16_bits.h).
// ---------------------------------------------------------------------------
template <int KIND>
struct Traits;
template <>
struct Traits<KIND_F32_F32> {
  using S = uint32_t;
  using D = uint32_t;
};
template <>
struct Traits<KIND_BF16_F32> {
  using S = uint16_t;
  using D = uint32_t;
};
template <>
struct Traits<KIND_F32_BF16> {
  using S = uint32_t;
  using D = uint16_t;
};
template <>
struct Traits<KIND_BF16_BF16> {
  using S = uint16_t;
  using D = uint16_t;
};

template <int KIND>
__device__ __forceinline__ uint32_t convert_one(uint32_t x) {
  if constexpr (KIND == KIND_BF16_F32) return bf16_to_f32_bits(x);
  else if constexpr (KIND == KIND_F32_BF16) return f32_to_bf16_bits(x);
  else return x;
}

// Destination element k of an item, written alone: source element k from the
// stage (cast), or +0 past n_copy.
template <int KIND>
__device__ __forceinline__ void scalar_elem(const uint8_t *stage, int lead, char *dst, int k, int n_copy) {
  using S = typename Traits<KIND>::S;
  using D = typename Traits<KIND>::D;
  uint32_t v = 0;
  if (k < n_copy) v = convert_one<KIND>((uint32_t)*reinterpret_cast<const S *>(stage + lead + k * (int)sizeof(S)));
  reinterpret_cast<D *>(dst)[k] = (D)v;
}

// The staged source of an item: the aligned 16-byte blocks that hold its
// valid source bytes [src, src + src_bytes).  `lead` is the offset of the
// first source byte in its block (a multiple of the element size), so stage
// byte lead + b holds source byte b.  Every staged byte shares a 16-byte
// block, and so a page, with a valid source byte: the widened read stays in
// mapped memory, and sources are never written during a call.
struct Staged {
  int lead, bytes;
};

__device__ __forceinline__ Staged staged_of(const char *src, int src_bytes) {
  Staged st;
  st.lead = (int)((uint32_t)(uintptr_t)src & 15u);
  st.bytes = src_bytes > 0 ? (st.lead + src_bytes + 15) & ~15 : 0;
  return st;
}

// What the producer tells the consumers about the item in a stage: written to
// shared memory before the stage's "full" barrier is armed, so consumers read
// it from shared memory after their wait instead of going back to global
// memory for the work item.
struct StageHeader {
  const char *src;  // first source element of the item
  char *dst;        // first destination element
  int32_t n_copy;
  int32_t n_total;
  int32_t kind;     // kSkipItem: nothing to do (refused by the producer)
  int32_t reserved;
};
static_assert(sizeof(StageHeader) <= kHeaderBytes, "stage header too large");
static_assert(sizeof(StageHeader) == 32, "the prefetch table holds 32-byte headers");

// Warm L2 with the staged source of the item with header h -- the 16-byte
// blocks its bulk copy will read -- without waiting for it.  A prefetch is
// only a hint into L2, which every SM sees coherently, so it may be issued
// before the previous kernel on the stream has finished: the bulk copy after
// griddepcontrol.wait still reads whatever that kernel wrote.  Issued by a
// launch whose blocks start while the previous launch drains, it puts the
// first reads in flight during that tail instead of after it.  A CTA whose
// whole work fits the ring prefetches its first item only.  Measured on one
// GB300, prefetching three or four such items made launches slower when
// nothing overlaps (behind a kernel that does not release its dependents
// early); the first item alone gained back to back and behind such kernels.
__device__ __forceinline__ void prefetch_item(const StageHeader &h) {
  const int ss = (h.kind & 1) ? 2 : 4;
  const Staged st = staged_of(h.src, h.n_copy * ss);
  if (st.bytes > 0 && st.bytes <= kStagedMax)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(h.src - st.lead), "r"((uint32_t)st.bytes)
                 : "memory");
}
constexpr int32_t kSkipItem = -1;
constexpr int32_t kDoneItem = -2;  // no item follows: the consumers leave

// The work-sharing word: bits 0..23 count the items handed out since the
// word was taken, bits 24..39 count the CTAs taking items from it ("users"),
// bits 40..63 hold the tag of the launch that took it (0: never taken).
//   * A CTA joins after its fixed-order items.  If the word carries its own
//     launch's tag, it adds itself as a user, and stays one if the tag is
//     still its own in the value the add returns (else it undoes the add).
//     If the word has no users, the CTA takes it for its launch with one
//     compare-and-swap: its tag, one user, count 0.  If another launch's
//     CTAs are using it, the CTA does not join.
//   * A user takes item fixed_rounds*G + (count before its add) by adding 1,
//     and leaves (removes itself as a user) on the first index past the end.
//   * A CTA that does not join takes the rest of its fixed order,
//     b + m*G for m >= fixed_rounds.
// Only the launch holding the word adds to its count, and the word changes
// hands only while it has no users, which happens after every user saw the
// end of the count: so when any CTA of a launch joins, that launch's users
// take every shared item between them; when none joins, the fixed order
// covers them.  A CTA that does not join may repeat items a user took; the
// second copy writes the same bytes, as every item's output depends on the
// inputs only.  Launches of one layout that overlap on the GPU (different
// streams) therefore give the same results as launches in turn.  The host
// keeps the shared part below 2^22 items so the count never reaches bit 24.
constexpr unsigned long long kSchedUser = 1ull << 24;
constexpr unsigned long long kSchedCountMask = kSchedUser - 1;
__device__ __forceinline__ uint32_t sched_tag_of(unsigned long long v) { return (uint32_t)(v >> 40); }
__device__ __forceinline__ uint32_t sched_users_of(unsigned long long v) { return (uint32_t)(v >> 24) & 0xFFFFu; }

__device__ __forceinline__ unsigned long long load_relaxed(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __noinline__ bool sched_join(unsigned long long *word, uint32_t tag) {
  unsigned long long v = load_relaxed(word);
  for (int attempt = 0; attempt < 4; ++attempt) {
    if (sched_tag_of(v) == tag) {
      const unsigned long long r = atomicAdd(word, kSchedUser);
      if (sched_tag_of(r) == tag) return true;
      atomicAdd(word, 0ull - kSchedUser);  // taken by another launch meanwhile
      return false;
    }
    if (sched_users_of(v) != 0) return false;
    const unsigned long long c = atomicCAS(word, v, ((unsigned long long)tag << 40) | kSchedUser);
    if (c == v) return true;
    v = c;
  }
  return false;
}

// Consumer side of one item.  `stage` holds the item's staged source.
// `ct` is the consumer thread index in [0, kConsumers).  Each thread handles
// kBatch destination vectors per round: it reads all their source words from
// shared memory first, then converts and stores them.
constexpr int kBatch = 1;

template <int KIND>
__device__ __forceinline__ void consume_item(const char *src, char *dst, int n_copy, int n_total,
                                             const uint8_t *stage, int ct) {
  using S = typename Traits<KIND>::S;
  using D = typename Traits<KIND>::D;
  constexpr int DU = 16 / (int)sizeof(D);      // elements per destination vector
  constexpr int SW = DU * (int)sizeof(S) / 4;  // source words per vector (2, 4 or 8)
  const int lead = (int)((uint32_t)(uintptr_t)src & 15u);

  // Destination: scalar head to the first 16-byte boundary, vectors, tail.
  int h = (int)(((16u - ((uint32_t)(uintptr_t)dst & 15u)) & 15u) / sizeof(D));
  h = h < n_total ? h : n_total;
  const int nvec = (n_total - h) / DU;
  const int tail0 = h + nvec * DU;
  if (ct < h) scalar_elem<KIND>(stage, lead, dst, ct, n_copy);
  if (tail0 + ct < n_total) scalar_elem<KIND>(stage, lead, dst, tail0 + ct, n_copy);

  // Every vector's source starts at the same byte phase inside a stage word
  // (vectors are SW words apart).  When that phase is zero and the first
  // vector's word is aligned to the load width, every vector's source is SW
  // whole words read with 8- or 16-byte loads and no shift ("wide").
  const int rb = ((lead + h * (int)sizeof(S)) & 3) * 8;
  constexpr int WA = SW < 4 ? SW : 4;  // words per wide load
  const bool wide = rb == 0 && (((lead + h * (int)sizeof(S)) >> 2) % WA) == 0;
  const uint32_t *stage32 = reinterpret_cast<const uint32_t *>(stage);
  for (int base = ct; base < nvec; base += kBatch * kConsumers) {
    uint32_t wv[kBatch][SW + 1];
    int mode[kBatch];  // 0 none, 1 whole vector, 2 all padding, 3 element by element (valid then padding)
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = base + b * kConsumers;
      const int e0 = h + j * DU;
      mode[b] = j >= nvec ? 0 : e0 >= n_copy ? 2 : e0 + DU <= n_copy ? 1 : 3;
      if (mode[b] == 1) {
        const int wi = (lead + e0 * (int)sizeof(S)) >> 2;
        if (wide) {
          if constexpr (SW == 2) {
            const uint2 t = *reinterpret_cast<const uint2 *>(stage32 + wi);
            wv[b][0] = t.x;
            wv[b][1] = t.y;
          } else {
#pragma unroll
            for (int q = 0; q < SW / 4; ++q) {
              const uint4 t = *reinterpret_cast<const uint4 *>(stage32 + wi + 4 * q);
              wv[b][4 * q + 0] = t.x;
              wv[b][4 * q + 1] = t.y;
              wv[b][4 * q + 2] = t.z;
              wv[b][4 * q + 3] = t.w;
            }
          }
          wv[b][SW] = 0;
        } else {
#pragma unroll
          for (int k = 0; k <= SW; ++k) wv[b][k] = stage32[wi + k];
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int e0 = h + (base + b * kConsumers) * DU;
      uint4 *d = reinterpret_cast<uint4 *>(dst + e0 * (int)sizeof(D));
      if (mode[b] == 1) {
        uint32_t sw[SW];
#pragma unroll
        for (int k = 0; k < SW; ++k) sw[k] = wide ? wv[b][k] : __funnelshift_r(wv[b][k], wv[b][k + 1], rb);
        uint32_t o[4];
        if constexpr (KIND == KIND_BF16_F32) {
          o[0] = sw[0] << 16;
          o[1] = sw[0] & 0xFFFF0000u;
          o[2] = sw[1] << 16;
          o[3] = sw[1] & 0xFFFF0000u;
        } else if constexpr (KIND == KIND_F32_BF16) {
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = f32_to_bf16_bits(sw[2 * i]) | (f32_to_bf16_bits(sw[2 * i + 1]) << 16);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = sw[i];
        }
        store_vec(d, o[0], o[1], o[2], o[3]);
      } else if (mode[b] == 2) {
        store_vec(d, 0u, 0u, 0u, 0u);
      } else if (mode[b] == 3) {
#pragma unroll 1
        for (int e = 0; e < DU; ++e) scalar_elem<KIND>(stage, lead, dst, e0 + e, n_copy);
      }
    }
  }
}

// The header of work item w as the consumers read it: its source and
// destination pointers resolved from the launch's slots (`base` is the slot
// base of its layout).  Reads only the parameter block.
template <class Args>
__device__ __forceinline__ StageHeader resolve_item(const Args &a, const WorkItem &w, int32_t base) {
  const int ss = (w.kind & 1) ? 2 : 4, ds = (w.kind & 2) ? 2 : 4;
  StageHeader h;
  h.src = reinterpret_cast<const char *>(a.slot[base + w.src_slot]) + w.src_off * (int64_t)ss;
  h.dst = reinterpret_cast<char *>(const_cast<void *>(a.slot[base + w.dst_slot])) + w.dst_off * (int64_t)ds;
  h.n_copy = w.n_copy;
  h.n_total = w.n_total;
  h.kind = w.kind;
  h.reserved = 0;
  return h;
}

template <class Args>
__global__ void __launch_bounds__(kThreads, 3) walk_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageStride);
  uint64_t *empty = full + kStages;
  StageHeader *pre = reinterpret_cast<StageHeader *>(smem + kPrefetchOffset);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  allow_next_grid();
  __syncthreads();

  const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
  if (warp == 0) {
    const int64_t G = gridDim.x, n = a.n_items;
    const Sched sc = a.sched;
    const int64_t shared0 = sc.word ? sc.fixed_rounds * G : 0;  // first shared item
    // This CTA's fixed-order items are blockIdx.x + m * G below fixed_end (at
    // least one: the grid is at most n, and a launch that shares items keeps
    // at least one fixed round).  Prologue, before waiting for the previous
    // kernel: in a single launch of at most kPrologueMaxRounds items per CTA,
    // the warp's lanes resolve the first n_pre of them at once -- descriptor
    // from the work table, source and destination pointers from the
    // parameter block -- into `pre`.  Done by one thread, each item's lookups
    // are a chain of dependent loads that miss the caches on a fresh launch,
    // and the chain would sit between consecutive bulk copies.  A long
    // launch keeps its pipeline full anyway and loses more by starting late
    // (every lane's lookups must land before the first copy); a batched one
    // resolves items one at a time (see BatchArgs).
    const int64_t fixed_end = sc.word ? (shared0 < n ? shared0 : n) : n;
    const int64_t n_fixed = (int64_t)blockIdx.x < fixed_end ? (fixed_end - blockIdx.x + G - 1) / G : 0;
    int n_pre = Args::kParallelPrologue && n <= kPrologueMaxRounds * G
                    ? (int)(n_fixed < kPrefetch ? n_fixed : kPrefetch) : 0;
    if (n_pre > 0) {
      if (lane < n_pre) {
        int cur = 0;
        int32_t base = 0;
        const WorkItem w = a.fetch(blockIdx.x + (int64_t)lane * G, &base, &cur);
        const StageHeader h = resolve_item(a, w, base);
        pre[lane] = h;
        if (lane < (n_fixed > kStages ? kL2PrefetchItems : 1)) prefetch_item(h);
      }
      __syncwarp();
    }
    // Without the parallel prologue, lane 0 resolves the items that fill the
    // ring first (at least item 0: blockIdx.x in every schedule, the grid
    // being at most n) one by one into `pre`, also before waiting for the
    // previous kernel on the stream, and prefetches their sources (item 0's
    // alone in a CTA whose whole work fits the ring).
    int cursor = 0;  // layout of the last fetched item (batched launches; lane 0's walk)
    if (n_pre == 0) {
      const int64_t depth = n >= kSeqPrefetchMinRounds * G ? kL2PrefetchItems : 1;
      const int n_seq = (int)(n_fixed < depth ? n_fixed : depth);
      if (lane == 0) {
        for (int mi = 0; mi < n_seq; ++mi) {
          int32_t base = 0;
          const WorkItem w = a.fetch(blockIdx.x + (int64_t)mi * G, &base, &cursor);
          pre[mi] = resolve_item(a, w, base);
          if (n_fixed > kStages || mi == 0) prefetch_item(pre[mi]);
        }
      }
      __syncwarp();
      n_pre = n_seq;
    }
    // First ring fill, in parallel: after the dependent-launch wait, lane s
    // stages the CTA's fixed-order item s into stage s itself (header, armed
    // barrier, bulk copy), so the first copies go out together instead of one
    // after another from the producer lane.  When more items follow, one
    // resolved header stays for the producer's loop to start from: a CTA that
    // shares its last items keeps one fixed-order item for its claim loop,
    // and one whose later descriptors are fetched one ahead keeps the last
    // resolved one.
    int n_first = 0;
    bool skip0 = false;
    {
      const int64_t avail = sc.word ? n_fixed - 1 : n_fixed;
      const int64_t keep = sc.word || n_pre < n_fixed ? n_pre - 1 : n_pre;
      const int64_t nf = avail < keep ? avail : keep;
      n_first = nf < kStages ? (int)(nf > 0 ? nf : 0) : kStages;
      if (n_first > 0) {
        wait_for_previous_grid();
        if (lane < n_first) {
          const StageHeader h = pre[lane];
          if (lane == 0 && blockIdx.x == 0 && (a.fault & kFaultSkipFirstStage)) {
            skip0 = true;
          } else {
            const Staged st = staged_of(h.src, h.n_copy * ((h.kind & 1) ? 2 : 4));
            uint32_t bytes = (uint32_t)st.bytes;
            StageHeader *hd = reinterpret_cast<StageHeader *>(smem + lane * kStageStride + kStageDataBytes);
            *hd = h;
            if (bytes > (uint32_t)kStagedMax) {  // never planned; the consumers skip it
              atomicOr(a.status, kStatusBadItem);
              hd->kind = kSkipItem;
              bytes = 0;
            }
            mbar_arrive_expect_tx(&full[lane], bytes);
            if (bytes) bulk_copy_g2s(smem + lane * kStageStride, h.src - st.lead, bytes, &full[lane]);
          }
        }
        __syncwarp();
      }
    }
    if (lane != 0) return;
    // Producer (lane 0).  Item indices are claimed two items ahead of use,
    // and the descriptors of items past the prefetched ones are fetched one
    // ahead, so neither the work-sharing word's round trip nor a descriptor
    // load sits on a stage hand-off: issue() starts a claim without looking
    // at what a shared claim's atomic add returns, and take() turns it into
    // an index one item later.
    // part 0: fixed-order items; 1: user of the word; 2: fixed order over
    // [shared0, n); 3: nothing left.
    int part = sc.word ? 0 : 2;
    int64_t m = 0;
    struct Claim {
      unsigned long long v;  // an item index, or the word's value before a shared claim's add
      int32_t pm;            // >= 0: the item's resolved header is pre[pm]
      bool shared;
    };
    auto issue = [&]() -> Claim {
      if (part == 0) {
        if (m < sc.fixed_rounds) {
          const int64_t mm = m++;
          return Claim{(unsigned long long)(blockIdx.x + mm * G), mm < n_pre ? (int32_t)mm : -1, false};
        }
        m = 0;
        const bool mixed_out = (sc.flags & kSchedMixed) && (blockIdx.x & 1u);
        part = !mixed_out && sched_join(sc.word, sc.tag) ? 1 : 2;
      }
      if (part == 1) return Claim{atomicAdd(sc.word, 1ull), -1, true};
      if (part == 2) return Claim{(unsigned long long)(shared0 + blockIdx.x + (m++) * G), -1, false};
      return Claim{(unsigned long long)n, -1, false};
    };
    // Claims resolve in the order they were issued.  Shared counts only grow
    // while this CTA is a user, so after the first shared claim past the end
    // every later one is past it too; the CTA leaves on the first.  Its adds
    // issued before the leave come first in the word's order (one thread,
    // one address), so the leave never lands ahead of them.
    auto take = [&](Claim q) -> int64_t {
      if (!q.shared) return (int64_t)q.v;
      const int64_t i = shared0 + (int64_t)(q.v & kSchedCountMask);
      if (i < n) return i;
      if (part == 1) {
        atomicAdd(sc.word, 0ull - kSchedUser);  // leave
        part = 3;
      }
      return n;
    };
    int64_t k = n_first;  // stages armed so far
    bool skipped_first = skip0, stopped = false;
    // Stage the item with resolved header h in the ring; false if the stage
    // never came free (the wait gave up).
    auto stage_item = [&](const StageHeader &h) -> bool {
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u, a.wait_limit_ns)) {
        atomicOr(a.status, kStatusProducerWait);
        return false;
      }
      if (k == 0 && blockIdx.x == 0 && (a.fault & kFaultSkipFirstStage)) {
        skipped_first = true;
        ++k;
        return true;
      }
      const int ss = (h.kind & 1) ? 2 : 4;
      const Staged st = staged_of(h.src, h.n_copy * ss);
      uint32_t bytes = (uint32_t)st.bytes;
      StageHeader *hd = reinterpret_cast<StageHeader *>(smem + s * kStageStride + kStageDataBytes);
      *hd = h;
      if (bytes > (uint32_t)kStagedMax) {  // never planned; the consumers skip it
        atomicOr(a.status, kStatusBadItem);
        hd->kind = kSkipItem;
        bytes = 0;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      if (bytes) bulk_copy_g2s(smem + s * kStageStride, h.src - st.lead, bytes, &full[s]);
      ++k;
      return true;
    };
    const StageHeader h0 = pre[0];
    wait_for_previous_grid();
    if (!sc.word) {
      // Fixed order: items blockIdx.x + mi * G; past the prefetched ones,
      // each descriptor is fetched one item ahead.
      WorkItem nxt{};
      int32_t nxt_base = 0;
      for (int64_t mi = n_first, i = blockIdx.x + mi * G; i < n; i += G, ++mi) {
        const StageHeader h = mi == 0 ? h0 : mi < n_pre ? pre[mi] : resolve_item(a, nxt, nxt_base);
        if (mi + 1 >= n_pre && i + G < n) nxt = a.fetch(i + G, &nxt_base, &cursor);
        if (!stage_item(h)) {
          stopped = true;
          break;
        }
      }
    } else {
      // Shared: each round issues the claim two items ahead and takes the
      // one issued the round before (a first round only primes that queue).
      // Item c0 is in hand: item 0's header h0 (c0_pm == -2), a prefetched
      // header (c0_pm >= 0) or a fetched descriptor (c0_pm == -1).  Joining
      // the word comes after the wait above, when an earlier launch of the
      // same operation on the stream has let go of it.
      m = 1 + n_first;
      int64_t c0 = blockIdx.x + n_first * G;
      int32_t c0_pm = n_first > 0 ? n_first : -2, c0_base = 0;
      WorkItem c0_w{};
      Claim q1{};
      bool primed = false;
      while (c0 < n) {
        const Claim qn = issue();
        if (!primed) {
          q1 = qn;
          primed = true;
          continue;
        }
        const StageHeader h = c0_pm == -2 ? h0 : c0_pm >= 0 ? pre[c0_pm] : resolve_item(a, c0_w, c0_base);
        const int64_t c1 = take(q1);
        if (c1 < n) {
          c0_pm = q1.pm;
          if (c0_pm < 0) c0_w = a.fetch(c1, &c0_base, &cursor);
        }
        q1 = qn;
        c0 = c1;
        if (!stage_item(h)) {
          stopped = true;
          break;
        }
      }
    }
    if (part == 1) atomicAdd(sc.word, 0ull - kSchedUser);  // stopped early: leave
    // Leave no bulk copy in flight when this thread exits: wait for the last
    // armed phase of every stage (consumers may have left early).  This comes
    // before the end marker below, which completes one more phase of a stage.
    for (int64_t kk = k > kStages ? k - kStages : 0; kk < k; ++kk) {
      if (kk == 0 && skipped_first) continue;
      if (!mbar_wait(&full[kk % kStages], (uint32_t)(kk / kStages) & 1u, a.wait_limit_ns))
        atomicOr(a.status, kStatusDrainWait);
    }
    // With a work-sharing word the consumers do not know their item count:
    // tell them that no item follows with a header of kind kDoneItem in the
    // next stage, its phase completed by a plain arrive.
    if (sc.word && !stopped) {
      const int s = (int)(k % kStages);
      const uint32_t round = (uint32_t)(k / kStages);
      if (round == 0 || mbar_wait(&empty[s], (round - 1) & 1u, a.wait_limit_ns)) {
        reinterpret_cast<StageHeader *>(smem + s * kStageStride + kStageDataBytes)->kind = kDoneItem;
        mbar_arrive(&full[s]);
      } else {
        atomicOr(a.status, kStatusProducerWait);
      }
    }
    return;
  }

  // Consumers: the items come in stage order.  In the fixed order CTA b's
  // items are b, b + G, ... below n; a launch that shares items ends each
  // CTA's stream with an end marker instead.
  wait_for_previous_grid();
  const int ct = (int)threadIdx.x - 32;
  const bool counted = a.sched.word == nullptr;
  int64_t i = blockIdx.x;
  for (int64_t k = 0; !counted || i < a.n_items; ++k, i += gridDim.x) {
    const int s = (int)(k % kStages);
    if (!mbar_wait(&full[s], (uint32_t)(k / kStages) & 1u, a.wait_limit_ns)) {
      if (lane == 0) atomicOr(a.status, kStatusConsumerWait);
      return;
    }
    const StageHeader hd = *reinterpret_cast<const StageHeader *>(smem + s * kStageStride + kStageDataBytes);
    if (hd.kind == kDoneItem) return;
    const uint8_t *stage = smem + s * kStageStride;
    switch (hd.kind) {
      case KIND_F32_F32: consume_item<KIND_F32_F32>(hd.src, hd.dst, hd.n_copy, hd.n_total, stage, ct); break;
      case KIND_BF16_F32: consume_item<KIND_BF16_F32>(hd.src, hd.dst, hd.n_copy, hd.n_total, stage, ct); break;
      case KIND_F32_BF16: consume_item<KIND_F32_BF16>(hd.src, hd.dst, hd.n_copy, hd.n_total, stage, ct); break;
      case KIND_BF16_BF16: consume_item<KIND_BF16_BF16>(hd.src, hd.dst, hd.n_copy, hd.n_total, stage, ct); break;
      default: break;  // refused item
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

// Slot capacities of the three kernel variants.  The largest keeps the
// parameter block under CUDA's 32,764-byte limit.
constexpr int kSlotsSmall = 64;
constexpr int kSlotsMedium = 512;
constexpr int kSlotsLarge = FSDP_MAX_PARAMS + 2;
static_assert(sizeof(LaunchArgs<kSlotsLarge>) <= 32764, "parameter block too large");

std::atomic<int32_t> g_fault{0};
std::atomic<int32_t> g_upload_fault{0};  // fsdp_debug_set_upload_fault
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<int32_t> g_sched_mode{FSDP_SCHEDULE_DEFAULT};  // fsdp_debug_set_schedule
std::atomic<int32_t> g_grid_cap{0};                         // fsdp_debug_set_grid_cap

// The grid a table-driven launch actually gets: the planned grid, cut to the
// test cap when one is set.
int64_t capped_grid(int64_t grid) {
  const int64_t cap = g_grid_cap.load(std::memory_order_relaxed);
  return cap > 0 && grid > cap ? cap : grid;
}

// A launch shares its last quarter of items when it has at least
// kSharedMinRounds items per CTA -- a batched launch when its layouts have
// that many on average; other launches keep the fixed order.  Measured on
// one GB300: sharing made large single groups 5-8 % faster (blocks on a few
// slow SMs no longer set the end) and a batch of eight large groups 9 %
// faster, but a batch of 24 small groups (864 items each) 3 % slower: its
// fixed order was already balanced, and each shared item costs an atomic
// round trip on one word.
constexpr int64_t kSharedMinRounds = 8;
constexpr int64_t kSharedMaxItems = int64_t(1) << 22;  // keeps the count below bit 24

// The schedule of one launch of n items on `grid` CTAs.  `word` is the
// operation's work-sharing word (nullptr: fixed order) and `epoch` the host
// counter its tags come from: tags run 1 .. 2^24 - 1 and wrap, so a tag is
// reused only after 16.7M launches on one word.
Sched make_sched(unsigned long long *word, std::atomic<uint32_t> *epoch, int64_t n, int64_t grid,
                 int64_t n_layouts = 1) {
  Sched sc{nullptr, 0, 0, 0};
  const int32_t mode = g_sched_mode.load(std::memory_order_relaxed);
  if (!word || !epoch || grid <= 0 || mode == FSDP_SCHEDULE_FIXED) return sc;
  int64_t rounds = 0;
  if (mode == FSDP_SCHEDULE_DEFAULT) {
    if (n < kSharedMinRounds * grid * n_layouts) return sc;
    rounds = (n / grid) * 3 / 4;
  }
  if (n - rounds * grid > kSharedMaxItems) rounds = (n - kSharedMaxItems + grid - 1) / grid;
  if (rounds < 1) rounds = 1;  // every CTA's first item comes in the fixed order
  sc.word = word;
  sc.fixed_rounds = rounds;
  sc.tag = epoch->fetch_add(1, std::memory_order_relaxed) % 0xFFFFFFu + 1u;
  sc.flags = mode == FSDP_SCHEDULE_MIXED ? kSchedMixed : 0;
  return sc;
}

template <int NSLOT>
fsdp_status_t launch_variant(const fsdp_layout *L, Op op, const void *const *ptrs, int n_ptrs,
                             cudaStream_t stream) {
  LaunchArgs<NSLOT> a;
  a.items = L->d_items + L->op[op].first;
  a.n_items = L->op[op].count;
  a.status = L->d_status;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.fault = g_fault.load(std::memory_order_relaxed);
  a.reserved = 0;
  const int64_t grid = capped_grid(L->op[op].grid);
  a.sched = make_sched(L->d_sched + op, &L->sched_epoch[op], a.n_items, grid);
  for (int k = 0; k < n_ptrs; ++k) a.slot[k] = ptrs[k];
  for (int k = n_ptrs; k < NSLOT; ++k) a.slot[k] = nullptr;
  // Programmatic stream serialization: this launch may be scheduled while the
  // previous kernel on the stream drains; the kernel waits for it before
  // touching memory (see wait_for_previous_grid).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&walk_kernel<LaunchArgs<NSLOT>>), args);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  clear_error();
  return FSDP_OK;
}

fsdp_status_t launch(const fsdp_layout *L, Op op, const void *const *ptrs, int n_ptrs, cudaStream_t stream) {
  if (L->op[op].count == 0) {
    clear_error();
    return FSDP_OK;
  }
  if (n_ptrs <= kSlotsSmall) return launch_variant<kSlotsSmall>(L, op, ptrs, n_ptrs, stream);
  if (n_ptrs <= kSlotsMedium) return launch_variant<kSlotsMedium>(L, op, ptrs, n_ptrs, stream);
  return launch_variant<kSlotsLarge>(L, op, ptrs, n_ptrs, stream);
}

// Several layouts' work in one launch (the *_batched entry points).  The
// largest variant leaves room for the per-layout table in the parameter block.
constexpr int kBatchSlotsLarge = 3840;
static_assert(sizeof(BatchArgs<kBatchSlotsLarge>) <= 32764, "batched parameter block too large");

template <int NSLOT>
fsdp_status_t batch_launch_variant(const fsdp_layout *const *Ls, int n, Op op, const void *const *ptrs, int n_ptrs,
                                   const int32_t *slot_base, cudaStream_t stream) {
  BatchArgs<NSLOT> a;
  int64_t total = 0;
  int groups = 0;
  for (int g = 0; g < n; ++g) {
    const int64_t c = Ls[g]->op[op].count;
    if (c == 0) continue;
    a.items[groups] = Ls[g]->d_items + Ls[g]->op[op].first;
    a.start[groups] = total;
    a.slot_base[groups] = slot_base[g];
    total += c;
    ++groups;
  }
  if (total == 0) {
    clear_error();
    return FSDP_OK;
  }
  a.start[groups] = total;
  a.n_groups = groups;
  a.n_items = total;
  a.status = Ls[0]->d_status;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.fault = g_fault.load(std::memory_order_relaxed);
  for (int k = 0; k < n_ptrs; ++k) a.slot[k] = ptrs[k];
  for (int k = n_ptrs; k < NSLOT; ++k) a.slot[k] = nullptr;
  const int64_t grid = capped_grid(total < Ls[0]->resident ? total : Ls[0]->resident);
  a.sched = make_sched(Ls[0]->d_sched + op, &Ls[0]->sched_epoch[op], total, grid, groups);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&walk_kernel<BatchArgs<NSLOT>>), args);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  clear_error();
  return FSDP_OK;
}

fsdp_status_t batch_launch(const fsdp_layout *const *Ls, int n, Op op, const void *const *ptrs, int n_ptrs,
                           const int32_t *slot_base, cudaStream_t stream) {
  if (n_ptrs <= kSlotsSmall) return batch_launch_variant<kSlotsSmall>(Ls, n, op, ptrs, n_ptrs, slot_base, stream);
  if (n_ptrs <= kSlotsMedium) return batch_launch_variant<kSlotsMedium>(Ls, n, op, ptrs, n_ptrs, slot_base, stream);
  return batch_launch_variant<kBatchSlotsLarge>(Ls, n, op, ptrs, n_ptrs, slot_base, stream);
}

}  // namespace

// ---------------------------------------------------------------------------
// Host-side argument checks (nothing is launched unless all pass), shared
// with reduce.cu.
// ---------------------------------------------------------------------------
fsdp_status_t check_layout(const fsdp_layout *L) {
  if (!L) return fail(FSDP_EINVAL, "layout is NULL");
  if (L->device < 0) return fail(FSDP_EINVAL, "layout was planned without a device table");
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (cur != L->device)
    return fail(FSDP_EINVAL, "current device " + std::to_string(cur) + " is not the layout's device " +
                                 std::to_string(L->device));
  return FSDP_OK;
}

std::string arg_name(const char *what, int64_t index) {
  return std::string(what) + (index >= 0 ? "[" + std::to_string(index) + "]" : "");
}

fsdp_status_t check_ptr(const void *p, int64_t bytes, int64_t align, const char *what, int64_t index) {
  if (bytes == 0) return FSDP_OK;
  if (!p) return fail(FSDP_EINVAL, arg_name(what, index) + " is NULL");
  if (((uintptr_t)p) % (uintptr_t)align)
    return fail(FSDP_EINVAL, arg_name(what, index) + " is not " + std::to_string(align) + "-byte aligned");
  return FSDP_OK;
}

namespace {

// Every walk_kernel instance may use kSmemBytes of dynamic shared memory
// (needed once that is above the 48 KB default).
template <class Args>
cudaError_t allow_smem() {
  return cudaFuncSetAttribute(reinterpret_cast<const void *>(&walk_kernel<Args>),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

// ---------------------------------------------------------------------------
// Allocation-free pack (fsdp_pack_reduce_scatter_noalloc).
//
// Some callers cannot allocate device memory at the point where they pack:
// code that runs while another component owns every byte of the device's
// memory budget, code inside an allocator or memory-pool callback (where a
// cudaMalloc would re-enter the allocator), and runtimes that forbid device
// allocation after start-up.  For them the pack can run with its scratch --
// the status word and the work table that the kernel walks -- in this
// file-scope array instead of memory from fsdp_plan_layout.  The array is part
// of the loaded module: every GPU that loads the library holds it until the
// process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr size_t kNoAllocTableOffset = 256;               // status word, padded
constexpr int64_t kNoAllocMaxItems = (int64_t)((kNoAllocScratchBytes - kNoAllocTableOffset) / sizeof(WorkItem));
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Per-device set-up, done once by the first call on that device: the device
// address of the array (in host code its name is only a host-side stand-in)
// and the resident grid size.
struct NoAllocDevice {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  unsigned char *scratch = nullptr;
  int64_t resident = 0;
};
NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];

void noalloc_setup(NoAllocDevice &nd, int dev) {
  int sms = 0, per_sm = 0;
  void *ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsSmall>>();
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsMedium>>();
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsLarge>>();
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, walk_kernel<LaunchArgs<kSlotsSmall>>, kThreads, kSmemBytes);
  nd.err = e;
  if (e == cudaSuccess) {
    nd.scratch = static_cast<unsigned char *>(ptr);
    nd.resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  }
}

template <int NSLOT>
fsdp_status_t noalloc_launch(const WorkItem *items, int64_t n_items, uint32_t *status, int64_t grid,
                             const void *const *ptrs, int n_ptrs, cudaStream_t stream) {
  LaunchArgs<NSLOT> a;
  a.items = items;
  a.n_items = n_items;
  a.status = status;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.fault = 0;
  a.reserved = 0;
  a.sched = Sched{nullptr, 0, 0, 0};  // fixed order: the array holds no work-sharing word
  for (int k = 0; k < n_ptrs; ++k) a.slot[k] = ptrs[k];
  for (int k = n_ptrs; k < NSLOT; ++k) a.slot[k] = nullptr;
  // No programmatic stream serialization here: the kernel reads its work
  // table before griddepcontrol.wait, and this table was just rewritten on
  // the stream.  With plain stream order the launch starts only after
  // everything before it on the stream, whatever that is, has finished.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  void *args[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&walk_kernel<LaunchArgs<NSLOT>>), args);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  clear_error();
  return FSDP_OK;
}

}  // namespace

fsdp_status_t device_setup(fsdp_layout *L) {
  int dev = -1, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsSmall>>();
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsMedium>>();
  if (e == cudaSuccess) e = allow_smem<LaunchArgs<kSlotsLarge>>();
  if (e == cudaSuccess) e = allow_smem<BatchArgs<kSlotsSmall>>();
  if (e == cudaSuccess) e = allow_smem<BatchArgs<kSlotsMedium>>();
  if (e == cudaSuccess) e = allow_smem<BatchArgs<kBatchSlotsLarge>>();
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, walk_kernel<LaunchArgs<kSlotsSmall>>, kThreads, kSmemBytes);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("device query failed: ") + cudaGetErrorString(e));
  const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  L->resident = resident;
  L->sms = sms;
  for (int op = 0; op < OP_COUNT; ++op) {
    int64_t g = L->op[op].count < resident ? L->op[op].count : resident;
    L->op[op].grid = (int32_t)(g > 0 ? g : 0);
  }
  // One allocation: a 64-byte header -- the status word at byte 0, one
  // work-sharing word per operation from byte 32 -- then the work table.
  constexpr size_t kHeader = 64;
  static_assert(32 + OP_COUNT * sizeof(unsigned long long) <= kHeader, "device header too small");
  const size_t table_bytes = L->items.size() * sizeof(WorkItem);
  if (g_upload_fault.load(std::memory_order_relaxed))
    return fail(FSDP_ENOMEM, "cudaMalloc of the work table: simulated failure (fsdp_debug_set_upload_fault)");
  void *mem = nullptr;
  e = cudaMalloc(&mem, kHeader + table_bytes);
  if (e != cudaSuccess)
    return fail(FSDP_ENOMEM, std::string("cudaMalloc of the work table: ") + cudaGetErrorString(e));
  L->d_status = reinterpret_cast<uint32_t *>(mem);
  L->d_sched = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(mem) + 32);
  L->d_items = reinterpret_cast<WorkItem *>(reinterpret_cast<char *>(mem) + kHeader);
  e = cudaMemset(mem, 0, kHeader);
  if (e == cudaSuccess && table_bytes)
    e = cudaMemcpy(L->d_items, L->items.data(), table_bytes, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(mem);
    L->d_status = nullptr;
    L->d_sched = nullptr;
    L->d_items = nullptr;
    return fail(FSDP_ECUDA, std::string("work table upload: ") + cudaGetErrorString(e));
  }
  L->device = dev;
  return FSDP_OK;
}

void device_release(fsdp_layout *L) {
  if (!L->d_status) return;
  int cur = -1;
  const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != L->device;
  if (switched) cudaSetDevice(L->device);
  cudaFree(L->d_status);
  if (switched) cudaSetDevice(cur);
  L->d_status = nullptr;
  L->d_sched = nullptr;
  L->d_items = nullptr;
}

}  // namespace fsdp

using namespace fsdp;

extern "C" {

fsdp_status_t fsdp_pack_reduce_scatter(const fsdp_layout_t *L, const void *const *grads,
                                       void *const *bucket_bufs, fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  const int P = (int)L->desc.size(), B = (int)L->bucket.size();
  if (P > 0 && !grads) return fail(FSDP_EINVAL, "grads is NULL");
  if (B > 0 && !bucket_bufs) return fail(FSDP_EINVAL, "bucket_bufs is NULL");
  for (int p = 0; p < P; ++p) {
    const int64_t sz = dtype_bytes(L->desc[p].grad_dtype);
    if ((st = check_ptr(grads[p], L->desc[p].numel * sz, sz, "grads", p)) != FSDP_OK) return st;
  }
  for (int b = 0; b < B; ++b) {
    const int64_t sz = dtype_bytes(L->bucket[b].dtype);
    if ((st = check_ptr(bucket_bufs[b], (int64_t)L->W * L->bucket[b].S * sz, sz, "bucket_bufs", b)) != FSDP_OK)
      return st;
  }
  const void *ptrs[kSlotsLarge];
  for (int p = 0; p < P; ++p) ptrs[p] = grads[p];
  for (int b = 0; b < B; ++b) ptrs[P + b] = bucket_bufs[b];
  return launch(L, OP_PACK, ptrs, P + B, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_allgather_copy_in(const fsdp_layout_t *L, const void *const *local_shards, void *ag_input,
                                     fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  const int P = (int)L->desc.size();
  if (P > 0 && !local_shards) return fail(FSDP_EINVAL, "local_shards is NULL");
  for (int p = 0; p < P; ++p) {
    const int64_t sz = dtype_bytes(L->desc[p].shard_dtype);
    if ((st = check_ptr(local_shards[p], L->param[p].chunk * sz, sz, "local_shards", p)) != FSDP_OK) return st;
  }
  if ((st = check_ptr(ag_input, L->S_ag, 16, "ag_input", -1)) != FSDP_OK) return st;
  const void *ptrs[kSlotsLarge];
  for (int p = 0; p < P; ++p) ptrs[p] = local_shards[p];
  ptrs[P] = ag_input;
  return launch(L, OP_COPY_IN, ptrs, P + 1, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_allgather_copy_out(const fsdp_layout_t *L, const void *ag_output, void *const *full_params,
                                      fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  const int P = (int)L->desc.size();
  if ((st = check_ptr(ag_output, (int64_t)L->W * L->S_ag, 16, "ag_output", -1)) != FSDP_OK) return st;
  if (P > 0 && !full_params) return fail(FSDP_EINVAL, "full_params is NULL");
  for (int p = 0; p < P; ++p) {
    const int64_t sz = dtype_bytes(L->desc[p].param_dtype);
    if ((st = check_ptr(full_params[p], L->desc[p].numel * sz, sz, "full_params", p)) != FSDP_OK) return st;
  }
  const void *ptrs[kSlotsLarge];
  ptrs[0] = ag_output;
  for (int p = 0; p < P; ++p) ptrs[1 + p] = full_params[p];
  return launch(L, OP_COPY_OUT, ptrs, P + 1, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_reduce_scatter_copy_out(const fsdp_layout_t *L, const void *const *reduced_rows,
                                           void *const *sharded_grads, fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  const int P = (int)L->desc.size(), B = (int)L->bucket.size();
  if (B > 0 && !reduced_rows) return fail(FSDP_EINVAL, "reduced_rows is NULL");
  if (P > 0 && !sharded_grads) return fail(FSDP_EINVAL, "sharded_grads is NULL");
  for (int b = 0; b < B; ++b) {
    const int64_t sz = dtype_bytes(L->bucket[b].dtype);
    if ((st = check_ptr(reduced_rows[b], L->bucket[b].S * sz, sz, "reduced_rows", b)) != FSDP_OK) return st;
  }
  for (int p = 0; p < P; ++p) {
    const int64_t sz = dtype_bytes(L->desc[p].shard_dtype);
    if ((st = check_ptr(sharded_grads[p], L->param[p].chunk * sz, sz, "sharded_grads", p)) != FSDP_OK) return st;
  }
  const void *ptrs[kSlotsLarge];
  for (int b = 0; b < B; ++b) ptrs[b] = reduced_rows[b];
  for (int p = 0; p < P; ++p) ptrs[B + p] = sharded_grads[p];
  return launch(L, OP_RS_COPY_OUT, ptrs, B + P, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Batched calls: several layouts' work in one launch.
// ---------------------------------------------------------------------------
static fsdp_status_t check_batch(const fsdp_layout_t *const *Ls, int32_t n) {
  if (n < 0) return fail(FSDP_EINVAL, "n_layouts < 0");
  if (n > kMaxBatch) return fail(FSDP_EUNSUPPORTED, "more than 64 layouts in one batch");
  if (n > 0 && !Ls) return fail(FSDP_EINVAL, "layouts is NULL");
  for (int32_t g = 0; g < n; ++g) {
    fsdp_status_t st = check_layout(Ls[g]);
    if (st != FSDP_OK) return st;
  }
  return FSDP_OK;
}

fsdp_status_t fsdp_pack_reduce_scatter_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                               const void *const *grads, void *const *bucket_bufs,
                                               fsdp_stream_t stream) {
  fsdp_status_t st = check_batch(layouts, n_layouts);
  if (st != FSDP_OK) return st;
  int64_t slots = 0, n_grads = 0, n_bufs = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    n_grads += (int64_t)layouts[g]->desc.size();
    n_bufs += (int64_t)layouts[g]->bucket.size();
  }
  slots = n_grads + n_bufs;
  if (slots > kBatchSlotsLarge) return fail(FSDP_EUNSUPPORTED, "more than 3840 pointers in one batch");
  if (n_grads > 0 && !grads) return fail(FSDP_EINVAL, "grads is NULL");
  if (n_bufs > 0 && !bucket_bufs) return fail(FSDP_EINVAL, "bucket_bufs is NULL");
  const void *ptrs[kBatchSlotsLarge];
  int32_t base[kMaxBatch];
  int64_t gi = 0, bi = 0, at = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    const fsdp_layout *L = layouts[g];
    base[g] = (int32_t)at;
    for (size_t p = 0; p < L->desc.size(); ++p, ++gi) {
      const int64_t sz = dtype_bytes(L->desc[p].grad_dtype);
      if ((st = check_ptr(grads[gi], L->desc[p].numel * sz, sz, "grads", gi)) != FSDP_OK) return st;
      ptrs[at++] = grads[gi];
    }
    for (size_t b = 0; b < L->bucket.size(); ++b, ++bi) {
      const int64_t sz = dtype_bytes(L->bucket[b].dtype);
      if ((st = check_ptr(bucket_bufs[bi], (int64_t)L->W * L->bucket[b].S * sz, sz, "bucket_bufs", bi)) != FSDP_OK)
        return st;
      ptrs[at++] = bucket_bufs[bi];
    }
  }
  return batch_launch(layouts, n_layouts, OP_PACK, ptrs, (int)at, base, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_allgather_copy_in_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                             const void *const *local_shards, void *const *ag_inputs,
                                             fsdp_stream_t stream) {
  fsdp_status_t st = check_batch(layouts, n_layouts);
  if (st != FSDP_OK) return st;
  int64_t n_shards = 0;
  for (int32_t g = 0; g < n_layouts; ++g) n_shards += (int64_t)layouts[g]->desc.size();
  if (n_shards + n_layouts > kBatchSlotsLarge) return fail(FSDP_EUNSUPPORTED, "more than 3840 pointers in one batch");
  if (n_shards > 0 && !local_shards) return fail(FSDP_EINVAL, "local_shards is NULL");
  if (n_layouts > 0 && !ag_inputs) return fail(FSDP_EINVAL, "ag_inputs is NULL");
  const void *ptrs[kBatchSlotsLarge];
  int32_t base[kMaxBatch];
  int64_t si = 0, at = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    const fsdp_layout *L = layouts[g];
    base[g] = (int32_t)at;
    for (size_t p = 0; p < L->desc.size(); ++p, ++si) {
      const int64_t sz = dtype_bytes(L->desc[p].shard_dtype);
      if ((st = check_ptr(local_shards[si], L->param[p].chunk * sz, sz, "local_shards", si)) != FSDP_OK) return st;
      ptrs[at++] = local_shards[si];
    }
    if ((st = check_ptr(ag_inputs[g], L->S_ag, 16, "ag_inputs", g)) != FSDP_OK) return st;
    ptrs[at++] = ag_inputs[g];
  }
  return batch_launch(layouts, n_layouts, OP_COPY_IN, ptrs, (int)at, base, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_allgather_copy_out_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                              const void *const *ag_outputs, void *const *full_params,
                                              fsdp_stream_t stream) {
  fsdp_status_t st = check_batch(layouts, n_layouts);
  if (st != FSDP_OK) return st;
  int64_t n_params = 0;
  for (int32_t g = 0; g < n_layouts; ++g) n_params += (int64_t)layouts[g]->desc.size();
  if (n_params + n_layouts > kBatchSlotsLarge) return fail(FSDP_EUNSUPPORTED, "more than 3840 pointers in one batch");
  if (n_layouts > 0 && !ag_outputs) return fail(FSDP_EINVAL, "ag_outputs is NULL");
  if (n_params > 0 && !full_params) return fail(FSDP_EINVAL, "full_params is NULL");
  const void *ptrs[kBatchSlotsLarge];
  int32_t base[kMaxBatch];
  int64_t pi = 0, at = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    const fsdp_layout *L = layouts[g];
    base[g] = (int32_t)at;
    if ((st = check_ptr(ag_outputs[g], (int64_t)L->W * L->S_ag, 16, "ag_outputs", g)) != FSDP_OK) return st;
    ptrs[at++] = ag_outputs[g];
    for (size_t p = 0; p < L->desc.size(); ++p, ++pi) {
      const int64_t sz = dtype_bytes(L->desc[p].param_dtype);
      if ((st = check_ptr(full_params[pi], L->desc[p].numel * sz, sz, "full_params", pi)) != FSDP_OK) return st;
      ptrs[at++] = full_params[pi];
    }
  }
  return batch_launch(layouts, n_layouts, OP_COPY_OUT, ptrs, (int)at, base, reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_reduce_scatter_copy_out_batched(const fsdp_layout_t *const *layouts, int32_t n_layouts,
                                                   const void *const *reduced_rows, void *const *sharded_grads,
                                                   fsdp_stream_t stream) {
  fsdp_status_t st = check_batch(layouts, n_layouts);
  if (st != FSDP_OK) return st;
  int64_t n_rows = 0, n_grads = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    n_rows += (int64_t)layouts[g]->bucket.size();
    n_grads += (int64_t)layouts[g]->desc.size();
  }
  if (n_rows + n_grads > kBatchSlotsLarge) return fail(FSDP_EUNSUPPORTED, "more than 3840 pointers in one batch");
  if (n_rows > 0 && !reduced_rows) return fail(FSDP_EINVAL, "reduced_rows is NULL");
  if (n_grads > 0 && !sharded_grads) return fail(FSDP_EINVAL, "sharded_grads is NULL");
  const void *ptrs[kBatchSlotsLarge];
  int32_t base[kMaxBatch];
  int64_t ri = 0, gi = 0, at = 0;
  for (int32_t g = 0; g < n_layouts; ++g) {
    const fsdp_layout *L = layouts[g];
    base[g] = (int32_t)at;
    for (size_t b = 0; b < L->bucket.size(); ++b, ++ri) {
      const int64_t sz = dtype_bytes(L->bucket[b].dtype);
      if ((st = check_ptr(reduced_rows[ri], L->bucket[b].S * sz, sz, "reduced_rows", ri)) != FSDP_OK) return st;
      ptrs[at++] = reduced_rows[ri];
    }
    for (size_t p = 0; p < L->desc.size(); ++p, ++gi) {
      const int64_t sz = dtype_bytes(L->desc[p].shard_dtype);
      if ((st = check_ptr(sharded_grads[gi], L->param[p].chunk * sz, sz, "sharded_grads", gi)) != FSDP_OK)
        return st;
      ptrs[at++] = sharded_grads[gi];
    }
  }
  return batch_launch(layouts, n_layouts, OP_RS_COPY_OUT, ptrs, (int)at, base,
                      reinterpret_cast<cudaStream_t>(stream));
}

fsdp_status_t fsdp_sync_status(const fsdp_layout_t *L, fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  uint32_t word = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&word, L->d_status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && word) e = cudaMemset(L->d_status, 0, sizeof(word));
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("status read: ") + cudaGetErrorString(e));
  if (word)
    return fail(FSDP_ETIMEOUT, "a bounded device wait gave up (status bits " + std::to_string(word) + ")");
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_pack_reduce_scatter_noalloc(const fsdp_layout_t *L, const void *const *grads,
                                               void *const *bucket_bufs, fsdp_stream_t stream) {
  if (!L) return fail(FSDP_EINVAL, "layout is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(FSDP_EUNSUPPORTED, "device ordinal above 63");
  if (L->device >= 0 && L->device != dev)
    return fail(FSDP_EINVAL, "current device is not the layout's device");
  const int P = (int)L->desc.size(), B = (int)L->bucket.size();
  if (P > 0 && !grads) return fail(FSDP_EINVAL, "grads is NULL");
  if (B > 0 && !bucket_bufs) return fail(FSDP_EINVAL, "bucket_bufs is NULL");
  fsdp_status_t st;
  for (int p = 0; p < P; ++p) {
    const int64_t sz = dtype_bytes(L->desc[p].grad_dtype);
    if ((st = check_ptr(grads[p], L->desc[p].numel * sz, sz, "grads", p)) != FSDP_OK) return st;
  }
  for (int b = 0; b < B; ++b) {
    const int64_t sz = dtype_bytes(L->bucket[b].dtype);
    if ((st = check_ptr(bucket_bufs[b], (int64_t)L->W * L->bucket[b].S * sz, sz, "bucket_bufs", b)) != FSDP_OK)
      return st;
  }
  const int64_t count = L->op[OP_PACK].count;
  if (count > kNoAllocMaxItems)
    return fail(FSDP_EUNSUPPORTED, "the pack needs " + std::to_string(count) +
                                       " work items; the no-alloc scratch holds at most " +
                                       std::to_string(kNoAllocMaxItems));
  NoAllocDevice &nd = g_noalloc_devices[dev];
  std::call_once(nd.once, noalloc_setup, std::ref(nd), dev);
  if (nd.err != cudaSuccess)
    return fail(FSDP_ECUDA, std::string("no-alloc scratch set-up: ") + cudaGetErrorString(nd.err));
  if (count == 0) {
    clear_error();
    return FSDP_OK;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t *status = reinterpret_cast<uint32_t *>(nd.scratch);
  WorkItem *table = reinterpret_cast<WorkItem *>(nd.scratch + kNoAllocTableOffset);
  e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(table, L->items.data() + L->op[OP_PACK].first, (size_t)count * sizeof(WorkItem),
                        cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("work table copy: ") + cudaGetErrorString(e));
  const int64_t grid = capped_grid(count < nd.resident ? count : nd.resident);
  const void *ptrs[kSlotsLarge];
  for (int p = 0; p < P; ++p) ptrs[p] = grads[p];
  for (int b = 0; b < B; ++b) ptrs[P + b] = bucket_bufs[b];
  if (P + B <= kSlotsSmall) return noalloc_launch<kSlotsSmall>(table, count, status, grid, ptrs, P + B, s);
  if (P + B <= kSlotsMedium) return noalloc_launch<kSlotsMedium>(table, count, status, grid, ptrs, P + B, s);
  return noalloc_launch<kSlotsLarge>(table, count, status, grid, ptrs, P + B, s);
}

void fsdp_debug_set_upload_fault(int32_t fail_upload) {
  g_upload_fault.store(fail_upload ? 1 : 0, std::memory_order_relaxed);
}

void fsdp_debug_set_wait_fault(int32_t fault, int64_t wait_limit_ns) {
  g_fault.store(fault, std::memory_order_relaxed);
  g_wait_limit_ns.store(wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : kDefaultWaitLimitNs,
                        std::memory_order_relaxed);
}

fsdp_status_t fsdp_debug_set_grid_cap(int32_t max_blocks) {
  if (max_blocks < 0) return fail(FSDP_EINVAL, "grid cap must be >= 0, got " + std::to_string(max_blocks));
  g_grid_cap.store(max_blocks, std::memory_order_relaxed);
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_debug_set_schedule(int32_t mode) {
  if (mode < FSDP_SCHEDULE_DEFAULT || mode > FSDP_SCHEDULE_MIXED)
    return fail(FSDP_EINVAL, "unknown schedule mode " + std::to_string(mode));
  g_sched_mode.store(mode, std::memory_order_relaxed);
  clear_error();
  return FSDP_OK;
}

}  // extern "C"
