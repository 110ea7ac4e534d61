// pa_prefill_tc128.cu - multi-token causal paged attention for fp16 / bf16
// caches on the 5th-generation tensor cores (tcgen05 + TMEM), head_dim 128,
// 128-key tiles.
//
// What it computes is pa_prefill's: query i of a sequence's n new tokens sits
// at position p = L - n + i and attends to positions 0 .. p, read through the
// block table ("PagedAttention: paging the KV cache", How it works: prefill
// writes into the blocks; "PagedAttention: Manage the Cache Without Moving the
// Sequence", The kernel must understand the mapping). The rows of one
// (sequence, KV head) are numbered r = i * g + j (query i, head j of the
// group), so the g heads of a KV head share every K/V tile.
//
// A CTA owns 256 such rows as two row tiles of 128 (one TMEM lane per row)
// and streams the sequence's K and V in tiles of 128 tokens:
//   S = Q K_t^T      tcgen05.mma M=128 N=128 K=16 (x8), Q and K K-major
//   P = exp2(S * scale*log2e - m)   online softmax, one row per thread
//   O += P V_t       tcgen05.mma M=128 N=128 K=16 (x8), P from TMEM, V MN-major
// TMEM: row tile q uses columns 256q .. 256q+127 for S, overwritten in place
// by P (each 32-column chunk of S holds its 32 keys' P: 16-bit pairs of the
// high parts, then the bf16 low parts), and 256q+128 .. 256q+255 for O. Each row tile has one S buffer, so the
// two tiles take turns on the tensor core: the MMA warp issues
//   PV(A, t), S(A, t+1), PV(B, t), S(B, t+1), ...
// and tile B's softmax of step t runs while the tensor core computes tile A's
// PV and next scores, and the other way round. In-order execution of one
// thread's MMAs makes S(A, t+1) overwrite P(A, t) only after PV(A, t) has read
// it. Scores come 128 keys at a time, the N at which an MMA runs at the tensor
// core's full rate.
//
// K and V tiles (32 KB each) stream through a ring of five shared-memory
// slots in the order K_0, V_0, K_1, V_1, ..., so the producer runs two tiles
// ahead of the MMAs. Warp 8 issues the TMA copies (one box of 64 head-dim
// elements x block piece per column half) and publishes each tile's mask of
// tokens with valid data; warp 9 issues the MMAs from one thread; warps 0-3
// and 4-7 run the two softmaxes (warp w owns TMEM lanes 32 (w % 4) ..), so
// every SM sub-partition alternates one warp of each.
//
// The running maximum rises only when a row's tile maximum passes it by more
// than 8 (log2 units); the softmax warp then rescales its rows of O in TMEM
// (the previous PV of its tile has completed: S was committed after it).
// fp16 P carries 11 significant bits and is used whole. bf16 P carries 8: a
// 64-key half of a tile keeps a low bf16 part as well (O += P_hi V + P_lo V,
// about 16 bits per weight) when, for some row of the warp, the half's weights
// sum to more than 1/8 of the row's normaliser so far; otherwise the high part
// alone is used. Every weight of an unsplit half then errs by at most
// 2^-9 * 1/8 = 2^-12 of its row's total, the bound of a whole fp16 P.
//
// Masking: keys past a row's position get p = 0; V rows of tokens without
// valid data (past the sequence's length, or of a block whose id is out of
// range) are zeroed in shared memory before PV reads them. Every wait is
// bounded by %globaltimer; a CTA that gives up sets PA_DEVERR_TIMEOUT, drains
// the copies and MMAs it has in flight (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kD = 128;        // head dim
constexpr int kRows = 128;     // query rows per row tile (TMEM lanes)
constexpr int kKeys = 128;     // tokens per K/V tile
constexpr int kSlots = 5;      // K/V ring slots (one K or V tile each)
constexpr int kMaskSlots = 8;  // per-tile valid-token masks in flight
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kLimitNs = 2000000000ull;
constexpr float kShareLimit = 0.125f;  // bf16: split P when a tile's weight passes this share

struct Smem {
  static constexpr uint32_t kHalf = kKeys * 128;       // 128 rows of 128 bytes: 16 KB
  static constexpr uint32_t kItem = 2 * kHalf;         // one K or V tile, [column half][row][128 B]
  static constexpr uint32_t kQTile = 2 * kRows * 128;  // one row tile of Q, same layout
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kRing = kQ + 2 * kQTile;
  static constexpr uint32_t kBar = kRing + kSlots * kItem;
  // full[kSlots], empty[kSlots], mask_full[kMaskSlots], s_full[2], p_full[2],
  // o_done[2], fin, q_full
  static constexpr uint32_t kNumBars = 2 * kSlots + kMaskSlots + 2 + 2 + 2 + 1 + 1;
  static constexpr uint32_t kMask = kBar + kNumBars * 8;        // 2 x uint64 per mask slot
  static constexpr uint32_t kVotes = kMask + kMaskSlots * 16;   // [row tile][parity][warp] u32
  static constexpr uint32_t kMisc = kVotes + 2 * 2 * 4 * 4;     // tmem base, abort flag
  static constexpr uint32_t kTotal = kMisc + 16 + 1024;         // + base-alignment slack
};
static_assert(Smem::kTotal <= 232448, "shared memory budget");
static_assert(Smem::kRing % 1024 == 0 && Smem::kItem % 1024 == 0, "128-byte swizzle atoms");

// 128 consecutive fp32 TMEM columns of this thread's lane: four loads, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
#define PA_LD32(OFF)                                                                              \
  asm volatile(                                                                                   \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"   \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"          \
      : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]),                  \
        "=r"(r[OFF + 4]), "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]),                  \
        "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]),                \
        "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15]),              \
        "=r"(r[OFF + 16]), "=r"(r[OFF + 17]), "=r"(r[OFF + 18]), "=r"(r[OFF + 19]),              \
        "=r"(r[OFF + 20]), "=r"(r[OFF + 21]), "=r"(r[OFF + 22]), "=r"(r[OFF + 23]),              \
        "=r"(r[OFF + 24]), "=r"(r[OFF + 25]), "=r"(r[OFF + 26]), "=r"(r[OFF + 27]),              \
        "=r"(r[OFF + 28]), "=r"(r[OFF + 29]), "=r"(r[OFF + 30]), "=r"(r[OFF + 31])               \
      : "r"(taddr + OFF))
  PA_LD32(0);
  PA_LD32(32);
  PA_LD32(64);
  PA_LD32(96);
#undef PA_LD32
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 packed 32-bit words into consecutive TMEM columns of this thread's lane
// (no wait: the caller waits once for all its stores).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Grid: (row-pair tiles, H_kv, N); x is taken in reverse so the tiles with the
// largest positions (most K/V) start first.
template <bool IS_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using S = Smem;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(sm);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int s = blockIdx.z;
  const int kvh = blockIdx.y;
  const int g = a.group;
  const int q0 = __ldg(a.q_start + s);
  const int n = __ldg(a.q_start + s + 1) - q0;
  const int L = __ldg(a.seq_lens + s);
  const int64_t cap = static_cast<int64_t>(a.max_blocks) * a.block_size;
  const int rows = n * g;
  const int row0 = (static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)) * 2 * kRows;
  if (n <= 0 || row0 >= rows) return;  // uniform: nothing to do
  if (n > L || L > cap) {              // the whole sequence is invalid
    if (threadIdx.x == 0 && kvh == 0 && row0 == 0) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    return;
  }
  // K/V tiles each row tile needs: up to its last row's position (0: no rows).
  // Row tile 1 holds later positions than row tile 0, so nt[1] >= nt[0] unless
  // it has no rows.
  int nt[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int first = row0 + q * kRows;
    if (first >= rows) {
      nt[q] = 0;
    } else {
      const int i_last = min((first + kRows - 1) / g, n - 1);
      nt[q] = (L - n + i_last) / kKeys + 1;
    }
  }
  const int ntiles = max(nt[0], nt[1]);

  const uint32_t bar = base + S::kBar;
  auto full = [&](int i) { return bar + 8u * i; };
  auto empty = [&](int i) { return bar + 8u * (kSlots + i); };
  auto mask_full = [&](int i) { return bar + 8u * (2 * kSlots + i); };
  auto s_full = [&](int q) { return bar + 8u * (2 * kSlots + kMaskSlots + q); };
  auto p_full = [&](int q) { return bar + 8u * (2 * kSlots + kMaskSlots + 2 + q); };
  auto o_done = [&](int q) { return bar + 8u * (2 * kSlots + kMaskSlots + 4 + q); };
  const uint32_t fin = bar + 8u * (2 * kSlots + kMaskSlots + 6);
  const uint32_t q_full = bar + 8u * (2 * kSlots + kMaskSlots + 7);  // Q rows in shared memory
  uint64_t* masks = reinterpret_cast<uint64_t*>(sm + S::kMask);
  volatile uint32_t* votes = reinterpret_cast<volatile uint32_t*>(sm + S::kVotes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kMisc);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(sm + S::kMisc + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int i = 0; i < kMaskSlots; ++i) mbar_init(mask_full(i), 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(s_full(q), 1);
      mbar_init(p_full(q), 4);
      mbar_init(o_done(q), 1);
    }
    mbar_init(fin, 1);
    mbar_init(q_full, kSoftmaxWarps);
    *abort = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {  // TMEM: per row tile, S/P then O
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     base + S::kMisc),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  const int64_t table_row = static_cast<int64_t>(s) * a.max_blocks;
  const int tpo = a.tok_per_op;  // tokens per box: min(block_size, 64), a power of two
  const int ops = kKeys / tpo;   // boxes per column half of a tile (<= 16)
  // The first global reads go out before the start-up barrier, so that their
  // latency overlaps the barrier set-up and the TMEM allocation: each softmax
  // thread's Q row, and the producer's block ids of tile 0.
  int id0 = -1;
  if (warp == kProducerWarp && lane < ops && lane * tpo < L)
    id0 = __ldg(a.block_tables + table_row + (lane * tpo) / a.block_size);
  if (warp < kSoftmaxWarps) {
    // Q rows into shared memory (K-major, 128-byte swizzle), one row per
    // softmax thread; the MMA warp waits on q_full before the first scores
    const int q = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int R = row0 + q * kRows + r;
    const uint4* src = nullptr;
    if (R < rows)
      src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                           ((static_cast<int64_t>(q0) + R / g) * a.num_q_heads +
                                            static_cast<int64_t>(kvh) * g + R % g) * kD);
    uint4 row[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) row[c] = src != nullptr ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t off = S::kQ + q * S::kQTile + (c >> 3) * S::kHalf + r * 128u +
                           (((c & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + off) = row[c];
    }
    fence_proxy_async_smem();  // the MMAs read Q through the async proxy
  }

  tc_fence_before();
  __syncthreads();  // barriers initialised, TMEM allocated, Q rows stored
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // bound of every wait that depends on a K/V tile arriving (the test hook can shorten it)
  const uint64_t wait_ns = PA_STAGE_WAIT_NS(a, kLimitNs);
  if (warp < kSoftmaxWarps && lane == 0) mbar_arrive(q_full);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    const int tpo_shift = __ffs(tpo) - 1;
    const int stop = a.test_stop_stage >= 0 && a.test_stop_stage < ntiles ? a.test_stop_stage : ntiles;
    // lane j < ops reads the block id of piece j of a tile; the ids of tile
    // t + 1 are requested while tile t is issued, so no tile waits on them
    auto read_id = [&](int t) {
      int id = -1;
      const int tok = t * kKeys + lane * tpo;
      if (lane < ops && tok < L) id = __ldg(a.block_tables + table_row + tok / a.block_size);
      return id;
    };
    int blk_next = stop > 0 ? id0 : -1;  // tile 0's ids, read before the start-up barrier
    int issued = 0;  // ring items (K or V tiles) issued
    bool ok = true;
    for (int t = 0; ok && t < stop; ++t) {
      const int t0 = t * kKeys;
      const int blk = blk_next;
      if (t + 1 < stop) blk_next = read_id(t + 1);
      int off = 0;
      bool valid = false;
      if (lane < ops && t0 + lane * tpo < L) {
        off = (t0 + lane * tpo) % a.block_size;
        valid = blk >= 0 && blk < a.num_blocks;
        if (!valid) atomicOr(a.err, PA_DEVERR_BLOCK_ID);
      }
      const uint32_t okmask = __ballot_sync(0xffffffffu, valid);
      // tokens with valid data (a piece with a good block id, below L): lane
      // i answers for tokens 32k + i, one ballot per k
      uint32_t mk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tok = 32 * k + lane;
        mk[k] = __ballot_sync(0xffffffffu, t0 + tok < L && ((okmask >> (tok >> tpo_shift)) & 1u));
      }
      if (lane == 0) {
        // the slot was last read for tile t - kMaskSlots, whose softmaxes have
        // finished: the ring holds at most two tiles ahead of the MMAs
        masks[2 * (t % kMaskSlots)] = static_cast<uint64_t>(mk[0]) | (static_cast<uint64_t>(mk[1]) << 32);
        masks[2 * (t % kMaskSlots) + 1] =
            static_cast<uint64_t>(mk[2]) | (static_cast<uint64_t>(mk[3]) << 32);
        mbar_arrive(mask_full(t % kMaskSlots));
      }
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {  // K_t, then V_t
        const int slot = issued % kSlots;
        if (issued >= kSlots &&
            !wait_or_abort(empty(slot), ((issued / kSlots) - 1) & 1, abort, wait_ns)) {
          if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
          ok = false;
          break;
        }
        if (lane == 0)
          mbar_arrive_expect_tx(full(slot), static_cast<uint32_t>(__popc(okmask)) * tpo * kD * 2u);
        __syncwarp();
        if (valid) {
          const uint32_t dst = base + S::kRing + slot * S::kItem + lane * tpo * 128u;
          const CUtensorMap* map = which == 0 ? &tmk : &tmv;
          tma_load_4d(dst, map, full(slot), 0, kvh, off, blk);
          tma_load_4d(dst + S::kHalf, map, full(slot), 64, kvh, off, blk);
        }
        ++issued;
      }
    }
    // copies in flight complete before the CTA frees its shared memory
    for (int i = (issued > kSlots ? issued - kSlots : 0); i < issued; ++i)
      mbar_wait_bounded(full(i % kSlots), (i / kSlots) & 1, kLimitNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = umma_idesc(IS_BF16, kRows, kKeys, false);
    constexpr uint32_t id_o = umma_idesc(IS_BF16, kRows, kD, true);
    // A descriptor's start address is its low 14 bits in 16-byte units and
    // shared memory stays below 256 KB, so an offset is a plain add.
    const uint64_t dq0 = umma_desc(base + S::kQ, 16, 1024);
    const uint64_t dring_k = umma_desc(base + S::kRing, 16, 1024);
    const uint64_t dring_v = umma_desc(base + S::kRing, S::kHalf, 1024);
    auto issue_s = [&](int q, int t) {  // S of row tile q over K_t (ring item 2t)
      const uint64_t dq = dq0 + ((q * S::kQTile) >> 4);
      const uint64_t dk = dring_k + ((((2 * t) % kSlots) * S::kItem) >> 4);
      const uint32_t d = tmem + q * 256u;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t o = (kk >> 2) * S::kHalf + (kk & 3) * 32u;
        umma(d, dq + (o >> 4), dk + (o >> 4), id_s, kk > 0 ? 1u : 0u);
      }
      umma_commit(s_full(q));
    };
    auto issue_pv = [&](int q, int t, bool split) {  // O += P V_t (ring item 2t + 1)
      const uint64_t dv = dring_v + ((((2 * t + 1) % kSlots) * S::kItem) >> 4);
      const uint32_t p_col = tmem + q * 256u;
      const uint32_t d = tmem + q * 256u + 128u;
      // keys 16kk .. 16kk + 15: chunk kk / 2, high parts at 32 (kk / 2) + 8 (kk % 2)
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)
        umma_tmem_a(d, p_col + 32u * (kk >> 1) + 8u * (kk & 1), dv + ((kk * 16u * 128u) >> 4),
                    id_o, (t > 0 || kk > 0) ? 1u : 0u);
      if (split) {  // low parts, 16 columns further on
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_tmem_a(d, p_col + 32u * (kk >> 1) + 8u * (kk & 1) + 16u,
                      dv + ((kk * 16u * 128u) >> 4), id_o, 1u);
      }
    };
    bool ok = true;
    if (lane == 0) {
      ok = wait_or_abort(q_full, 0, abort, wait_ns) && wait_or_abort(full(0), 0, abort, wait_ns);
      if (ok) {
        tc_fence_after();
        for (int q = 0; q < 2; ++q)
          if (nt[q] > 0) issue_s(q, 0);
        umma_commit(empty(0));  // K_0
      }
      for (int t = 0; ok && t < ntiles; ++t) {
        const int iv = 2 * t + 1;  // V_t
        const int ik = 2 * t + 2;  // K_{t+1}
        bool v_ready = false, k_ready = false;
        for (int q = 0; q < 2; ++q) {
          if (t >= nt[q]) continue;
          if (!v_ready) {
            ok = wait_or_abort(full(iv % kSlots), (iv / kSlots) & 1, abort, wait_ns);
            if (!ok) break;
            v_ready = true;
          }
          ok = wait_or_abort(p_full(q), t & 1, abort, wait_ns);
          if (!ok) break;
          tc_fence_after();
          bool split = false;
          if constexpr (IS_BF16) {
            const volatile uint32_t* v = votes + (q * 2 + (t & 1)) * 4;
            split = (v[0] | v[1] | v[2] | v[3]) != 0u;
          }
          issue_pv(q, t, split);
          if (t + 1 == nt[q]) umma_commit(o_done(q));
          if (t + 1 < nt[q]) {
            if (!k_ready) {
              ok = wait_or_abort(full(ik % kSlots), (ik / kSlots) & 1, abort, wait_ns);
              if (!ok) break;
              tc_fence_after();
              k_ready = true;
            }
            issue_s(q, t + 1);
          }
        }
        if (!ok) break;
        umma_commit(empty(iv % kSlots));               // V_t: every PV of step t issued
        if (k_ready) umma_commit(empty(ik % kSlots));  // K_{t+1}: every S of step t + 1 issued
      }
      if (!ok) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
      umma_commit(fin);  // arrives once every MMA issued above has completed
      mbar_wait_bounded(fin, 0, kLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int R = row0 + q * kRows + r;
    const int i = R / g;
    const bool row_ok = R < rows;
    const int pos = row_ok ? L - n + i : -1;  // last key this row sees
    const uint32_t lane_base = tmem + q * 256u + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_col = lane_base;         // S, then P
    const uint32_t o_col = lane_base + 128u;  // O
    const float sl = a.scale_log2;
    const bool pos_scale = sl > 0.f;
    float m = -INFINITY;  // running max, log2 units
    float l = 0.f;
    bool ok = true;
    const int my_tiles = nt[q];
    for (int t = 0; t < my_tiles; ++t) {
      if (!wait_or_abort(s_full(q), t & 1, abort, wait_ns)) { ok = false; break; }
      if (!wait_or_abort(mask_full(t % kMaskSlots), (t / kMaskSlots) & 1, abort, wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t vm0 = masks[2 * (t % kMaskSlots)];
      const uint64_t vm1 = masks[2 * (t % kMaskSlots) + 1];
      const int k0 = t * kKeys;
      const bool all_valid = vm0 == ~0ull && vm1 == ~0ull;
      const bool whole = __all_sync(0xffffffffu, all_valid && k0 + kKeys - 1 <= pos);
      // logits in log2 units are x * sl; with sl > 0 the max commutes with the
      // scaling and the scaling folds into the exponent's FMA. Both passes
      // below read S from TMEM, 64 columns at a time, and mask it the same way.
      const float fs = pos_scale ? sl : 1.f;
      auto load_half = [&](int h, float (&x)[64]) {
        tmem_ld64(s_col + 64 * h, x);
        if (!pos_scale) {
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] *= sl;
        }
        if (!whole) {
          const uint64_t w = h ? vm1 : vm0;
          const int kh = k0 + 64 * h;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const bool valid = (kh + c <= pos) && ((w >> c) & 1ull);
            x[c] = valid ? x[c] : -INFINITY;
          }
        }
      };
      // ---- pass 1: the tile's row maximum
      float mx = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float x[64];
        load_half(h, x);
        float t22[22];  // 64 -> 22 -> 8 -> 3 -> 1 with three-input maxima
#pragma unroll
        for (int c = 0; c < 21; ++c) t22[c] = max3(x[c], x[c + 21], x[c + 42]);
        t22[21] = x[63];
        float t8[8];
#pragma unroll
        for (int c = 0; c < 7; ++c) t8[c] = max3(t22[c], t22[c + 7], t22[c + 14]);
        t8[7] = t22[21];
        mx = max3(mx, max3(max3(t8[0], t8[1], t8[2]), max3(t8[3], t8[4], t8[5]), t8[6]), t8[7]);
      }
      mx *= fs;
      const bool grow = mx > m + 8.f;
      const float m_new = grow ? mx : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = grow ? fast_exp2(m - m_use) : 1.f;
      // the previous PV of this row tile completed before S was committed
      if (t > 0 && __any_sync(0xffffffffu, grow && m != -INFINITY)) {
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(o_col + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(o_col + c, o);
        }
      }
      m = m_new;
      // ---- pass 2: p = exp2(x * fs - m), 64 keys at a time. Each 32-key
      // chunk's P goes over its own S columns 32c .. 32c + 31: 16-bit pairs of
      // its high parts in the first 16. bf16: the low parts go in the last 16
      // when, for some row of the warp, this half's weights pass 1/8 of the
      // normaliser so far (l * alpha plus the halves done, at most the final
      // one); otherwise zeros, and those rows use the high parts alone. The
      // MMA warp runs the low-part pass when any warp of the row tile voted.
      const uint64_t fs2 = f2(fs, fs);
      const uint64_t nm2 = f2(-m_use, -m_use);
      float l_run = l * alpha;
      bool voted = false;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float x[64];
        load_half(h, x);
        uint64_t ps[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f pairs
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 e = f2_split(fma_f2(f2(x[c], x[c + 1]), fs2, nm2));
          x[c] = fast_exp2(e.x);
          x[c + 1] = fast_exp2(e.y);
          ps[(c >> 1) & 3] = add_f2(ps[(c >> 1) & 3], f2(x[c], x[c + 1]));
        }
        ps[0] = add_f2(ps[0], ps[1]);
        ps[2] = add_f2(ps[2], ps[3]);
        ps[0] = add_f2(ps[0], ps[2]);
        const float2 psum2 = f2_split(ps[0]);
        const float psum = psum2.x + psum2.y;
        l_run += psum;
        bool split = false;
        if constexpr (IS_BF16) split = __any_sync(0xffffffffu, psum > kShareLimit * l_run);
        voted = voted || split;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t hi[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) hi[j] = pack2<IS_BF16>(x[32 * cc + 2 * j], x[32 * cc + 2 * j + 1]);
          const uint32_t col = s_col + 64 * h + 32 * cc;
          tmem_st16u(col, hi);
          if constexpr (IS_BF16) {
            uint32_t lo[16];
            if (split) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float2 hh = unpack2<true>(hi[j]);
                const float2 d = f2_split(
                    sub_f2(f2(x[32 * cc + 2 * j], x[32 * cc + 2 * j + 1]), f2(hh.x, hh.y)));
                lo[j] = pack2<true>(d.x, d.y);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) lo[j] = 0u;
            }
            tmem_st16u(col + 16, lo);
          }
        }
      }
      // one vote per warp (votes alternate by tile parity, so a vote for t + 2
      // is written only after the MMA warp has read the one for t)
      if constexpr (IS_BF16) {
        if (lane == 0) votes[(q * 2 + (t & 1)) * 4 + wq] = voted ? 1u : 0u;
      }
      l = l_run;
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // tokens without valid data: zero their V rows so 0 * garbage never
      // enters O (the slot holds V_t until this tile's PVs have completed;
      // both row tiles write the same zeros)
      if (!all_valid) {
        const int iv = 2 * t + 1;
        if (!wait_or_abort(full(iv % kSlots), (iv / kSlots) & 1, abort, wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t vbase = S::kRing + (iv % kSlots) * S::kItem;
        for (int idx = r; idx < kKeys * 16; idx += kRows) {
          const int tok = idx >> 4;
          const int rem = idx & 15;
          const uint64_t w = tok < 64 ? vm0 : vm1;
          if (!((w >> (tok & 63)) & 1ull))
            *reinterpret_cast<uint4*>(sm + vbase + (rem >> 3) * S::kHalf + tok * 128u +
                                      ((rem & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(q));
    }
    if (!ok) {
      if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
    } else if (my_tiles > 0) {
      // ---- epilogue: O / l once this row tile's last PV has completed
      if (wait_or_abort(o_done(q), 0, abort, wait_ns)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t ob = row_ok ? ((static_cast<int64_t>(q0) + i) * a.num_q_heads +
                                     static_cast<int64_t>(kvh) * g + R % g) * kD
                                  : 0;
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(o_col + c, o);
          if (row_ok) {
            if (a.out_dtype == PA_F32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + ob + c);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv,
                                     o[4 * e + 3] * inv);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + ob + c);
              const bool bf = a.out_dtype == PA_BF16;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float lo = o[8 * e + 2 * h] * inv;
                  const float hi = o[8 * e + 2 * h + 1] * inv;
                  w[h] = bf ? pack2<true>(lo, hi) : pack2<false>(lo, hi);
                }
                dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
      } else if (lane == 0) {
        atomicOr(a.err, PA_DEVERR_TIMEOUT);
        *abort = 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool IS_BF16>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a, dim3 grid,
                   cudaStream_t st) {
  auto kern = prefill_tc_kernel<IS_BF16>;
  const int smem = static_cast<int>(Smem::kTotal);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc128(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                                 bool bf16, dim3 grid, cudaStream_t st) {
  return bf16 ? launch<true>(tk, tv, a, grid, st) : launch<false>(tk, tv, a, grid, st);
}

}  // namespace pa
