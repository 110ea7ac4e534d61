// pa_prefill_tc.cu - multi-token causal paged attention over FP8 (E4M3)
// caches on the 5th-generation tensor cores (tcgen05 + TMEM) for head_dim 128,
// 64-key tiles. (fp16 / bf16 caches run on pa_prefill_tc128.cu.)
//
// What it computes is pa_prefill's: query i of a sequence's n new tokens sits
// at position p = L - n + i and attends to positions 0 .. p, read through the
// block table ("PagedAttention: paging the KV cache", How it works: prefill
// writes into the blocks; "PagedAttention: Manage the Cache Without Moving the
// Sequence", The kernel must understand the mapping). The rows of one
// (sequence, KV head) are numbered r = i * g + j (query i, head j of the
// group), so the g heads of a KV head share every K/V tile.
//
// A CTA owns 256 such rows as two tiles A and B of 128 (one TMEM lane per row
// in each) and streams the sequence's K and V in tiles of 64 tokens, each used
// by both row tiles:
//   S_t  = Q K_t^T     tcgen05.mma M=128 N=64  K=128, Q and K K-major
//   P_t  = exp2(S_t * scale*log2e - m)   online softmax, one row per thread
//   O   += P_t V_t     tcgen05.mma M=128 N=128 K=64, V MN-major
// TMEM: row tile q uses columns 256q .. 256q+255 - S double-buffered in the
// first 128, O in the last 128. P never leaves tensor memory: the softmax
// writes P_t over its own S buffer (bf16/fp16 pairs, 32 columns per part) and
// the PV MMA takes its A operand from there; S_{t+2} reuses the buffer only
// after PV_t, in the MMA warp's issue order. Warps 0-3 run the softmax of tile A and warps 4-7
// that of tile B (warp w owns TMEM lanes 32 (w % 4) ..), so every SM
// sub-partition alternates two independent softmax warps; warp 8 issues the
// TMA copies of K/V tiles (one box of 64 head-dim elements x block piece per
// column half), warp 9 issues the MMAs from one thread. The MMA warp issues
// S_{t+1} of both tiles before waiting for their P_t, so the tensor core
// computes the next scores while the softmax works.
//
// The running maximum rises only when a row's maximum exceeds it by more than
// 8 (log2 units); then the softmax warp waits for the previous O update and
// rescales its rows of O in TMEM. p stays below 2^8. A bf16 P carries only 8
// significant bits, so for bf16 inputs P is split into a high and a low bf16
// part, O += P_hi V + P_lo V, keeping about 16 bits of each weight; an fp16 P
// (11 bits) is used whole.
//
// FP8 (E4M3) caches: the TMA ring holds the codes (one 128-byte line per token
// for K and for V); two converter warps widen each tile exactly to fp16 into a
// ring of four tiles in the 16-bit layout the MMAs read (one warp K, one V, zeroing
// V rows without valid data), and every MMA runs in fp16. A bf16 query row is
// stored as fp16 times a power of two that keeps its largest element below
// 2^14, undone in that row's logit scale; P is then fp16 and used whole. k_scale
// folds into the logit scale, v_scale multiplies the output.
//
// Masking: keys past a row's position get p = 0; V rows of tokens that hold no
// valid data (past the sequence's length, or of a block with an id out of
// range) are zeroed in shared memory before O += P V reads them. Every wait is
// bounded by %globaltimer; a CTA that gives up sets PA_DEVERR_TIMEOUT, drains
// what it has in flight (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kD = 128;            // head dim
constexpr int kRowsTc = 128;       // query rows per row tile (TMEM lanes)
constexpr int kQTiles = 2;         // row tiles per CTA
constexpr int kBn = 64;            // tokens per K/V tile
constexpr int kStagesTc = 4;       // tiles in flight in the TMA ring
constexpr int kSoftmaxWarps = 4 * kQTiles;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kConvWarp = kSoftmaxWarps + 2;  // FP8: warps kConvWarp (K) and kConvWarp + 1 (V)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kLimitTcNs = 2000000000ull;

template <bool FP8>
constexpr int tc_threads() {
  return (kSoftmaxWarps + 2 + (FP8 ? 2 : 0)) * 32;
}

// Shared memory. 16-bit caches: the TMA ring holds the K/V tiles the MMAs
// read (kStagesTc of kStage). FP8: the TMA ring holds code tiles (kLoadStages
// of kCodeTile) and the MMAs read a ring of kMmaTiles widened tiles.
template <bool FP8>
struct TcSmem {
  static constexpr uint32_t kHalf = kBn * 128;                  // 64 token rows of 128 bytes
  static constexpr uint32_t kQTile = 2 * kRowsTc * 128;         // 2 halves x 128 rows x 128 B
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kStage = 4 * kHalf;                 // K halves, then V halves
  static constexpr uint32_t kStages = kQ + kQTiles * kQTile;    // tiles the MMAs read
  // The K and V tiles the MMAs read sit as [column half][stage][64 rows][128 B],
  // so consecutive stages are adjacent rows of one operand.
  static constexpr uint32_t kHalfStride = kStagesTc * kHalf;    // between column halves
  static constexpr uint32_t kKRing = kStages;
  static constexpr uint32_t kVRing = kStages + 2 * kHalfStride;
  static constexpr int kLoadStages = FP8 ? 2 : kStagesTc;   // TMA ring
  static constexpr int kMmaTiles = FP8 ? 4 : kStagesTc;
  static constexpr uint32_t kCodeTile = 2 * kHalf;              // K codes, then V codes
  static constexpr uint32_t kCodes = kStages + kMmaTiles * kStage;
  static constexpr uint32_t kBar = kCodes + (FP8 ? kLoadStages * kCodeTile : 0);
  // kv_full[NS], kv_empty[NS], s_full[2 tiles][2], p_full[2 tiles][2],
  // o_done[2 tiles][2], final, and for FP8 conv_full[4], conv_empty[4].
  // p_full and o_done alternate by tile parity: a softmax warp may publish
  // P_{t+1} before the MMA warp waits for P_t, and waits on o_done only now and
  // then, so a single barrier could run two phases ahead of its waiter, where
  // parity waits alias.
  static constexpr uint32_t kNumBars = 2 * kStagesTc + 4 + 4 + 4 + 1 + 8;
  static constexpr uint32_t kMask = kBar + kNumBars * 8;        // uint64 per ring stage
  static constexpr uint32_t kConvMask = kMask + kStagesTc * 8;  // FP8: uint64 per widened tile
  static constexpr uint32_t kMisc = kConvMask + 4 * 8;          // tmem base, abort flag
  static constexpr uint32_t kTotal = kMisc + 16 + 1024;         // + base-alignment slack
};
static_assert(TcSmem<false>::kTotal <= 232448 && TcSmem<true>::kTotal <= 232448,
              "shared memory budget");

// Grid: (row-pair tiles, H_kv, N); x is taken in reverse so the tiles with the
// largest positions (most K/V) start first.
template <bool IS_BF16, bool FP8>
__global__ void __launch_bounds__(tc_threads<FP8>(), 1)
    prefill_tc_e4m3_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using S = TcSmem<FP8>;
  constexpr bool MB = IS_BF16 && !FP8;  // MMA operand type: E4M3 caches run in fp16
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
  const int row0 = (static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)) * kQTiles * kRowsTc;
  if (n <= 0 || row0 >= rows) return;  // uniform: nothing to do
  if (n > L || L > cap) {              // the whole sequence is invalid
    if (threadIdx.x == 0 && kvh == 0 && row0 == 0) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    return;
  }
  // K/V tiles each row tile needs: up to its last row's position (0: no rows)
  int nt[kQTiles];
#pragma unroll
  for (int q = 0; q < kQTiles; ++q) {
    const int first = row0 + q * kRowsTc;
    if (first >= rows) {
      nt[q] = 0;
    } else {
      const int i_last = min((first + kRowsTc - 1) / g, n - 1);
      nt[q] = (L - n + i_last) / kBn + 1;
    }
  }
  const int ntiles = max(nt[0], nt[1]);

  const uint32_t bar = base + S::kBar;
  auto kv_full = [&](int k) { return bar + 8u * k; };
  auto kv_empty = [&](int k) { return bar + 8u * (kStagesTc + k); };
  auto s_full = [&](int q, int b) { return bar + 8u * (2 * kStagesTc + 2 * q + b); };
  auto p_full = [&](int q, int b) { return bar + 8u * (2 * kStagesTc + 4 + 2 * q + b); };
  auto o_done = [&](int q, int b) { return bar + 8u * (2 * kStagesTc + 8 + 2 * q + b); };
  const uint32_t fin = bar + 8u * (2 * kStagesTc + 12);
  auto conv_full = [&](int b) { return bar + 8u * (2 * kStagesTc + 13 + b); };
  auto conv_empty = [&](int b) { return bar + 8u * (2 * kStagesTc + 17 + b); };
  constexpr int LS = S::kLoadStages;  // TMA ring stages
  constexpr int NB = S::kMmaTiles;  // FP8: widened tiles, tile t in buffer t % NB
  uint64_t* masks = reinterpret_cast<uint64_t*>(sm + S::kMask);
  uint64_t* conv_masks = reinterpret_cast<uint64_t*>(sm + S::kConvMask);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kMisc);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(sm + S::kMisc + 4);

  if (threadIdx.x == 0) {
    for (int k = 0; k < kStagesTc; ++k) {
      mbar_init(kv_full(k), 1);
      mbar_init(kv_empty(k), FP8 ? 2 : 1);  // FP8: released by both converter warps
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(conv_full(b), 2);
      mbar_init(conv_empty(b), 1);
    }
    for (int q = 0; q < kQTiles; ++q) {
      mbar_init(s_full(q, 0), 1);
      mbar_init(s_full(q, 1), 1);
      mbar_init(p_full(q, 0), 4);
      mbar_init(p_full(q, 1), 4);
      mbar_init(o_done(q, 0), 1);
      mbar_init(o_done(q, 1), 1);
    }
    mbar_init(fin, 1);
    *abort = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {  // TMEM: per row tile, S double buffer + O
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     base + S::kMisc),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // ---- Q rows into shared memory (K-major, 128-byte swizzle), one row per thread.
  // FP8 with bf16 q: the row becomes fp16 times 2^(13 - e), e the exponent of
  // its largest magnitude; q_scale is the factor the row's logits undo.
  float q_scale = 1.f;
  if (warp < kSoftmaxWarps) {
    const int q = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int R = row0 + q * kRowsTc + r;
    const int i = R / g;
    const uint4* src = nullptr;
    if (R < rows)
      src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                           ((static_cast<int64_t>(q0) + i) * a.num_q_heads +
                                            static_cast<int64_t>(kvh) * g + R % g) * kD);
    uint4 row[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) row[c] = src != nullptr ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    if constexpr (FP8 && IS_BF16) {
      float mx = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t w[4] = {row[c].x, row[c].y, row[c].z, row[c].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = unpack2<true>(w[h]);
          mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      const int e = max(static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127, -100);
      const float p = __uint_as_float(static_cast<uint32_t>(127 + 13 - e) << 23);  // 2^(13-e)
      q_scale = __uint_as_float(static_cast<uint32_t>(127 - 13 + e) << 23);        // 2^(e-13)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint32_t w[4] = {row[c].x, row[c].y, row[c].z, row[c].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 f = unpack2<true>(w[h]);
          w[h] = pack2<false>(f.x * p, f.y * p);
        }
        row[c] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t off = S::kQ + q * S::kQTile + (c >> 3) * (kRowsTc * 128u) + r * 128u +
                           (((c & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + off) = row[c];
    }
  }
  // the producer's first block-id read goes out before the start-up barrier
  const int64_t table_row = static_cast<int64_t>(s) * a.max_blocks;
  int id_next = -1;
  if (warp == kProducerWarp && lane < a.ops_per_stage && lane * a.tok_per_op < L)
    id_next = __ldg(a.block_tables + table_row + (lane * a.tok_per_op) / a.block_size);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // bound of every wait that depends on a K/V tile arriving (the test hook can shorten it)
  const uint64_t wait_ns = PA_STAGE_WAIT_NS(a, kLimitTcNs);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    const int tpo = a.tok_per_op;
    const int stop = a.test_stop_stage >= 0 && a.test_stop_stage < ntiles ? a.test_stop_stage : ntiles;
    // lane j < ops_per_stage reads the block id of piece j of a tile; the ids
    // of tile t + 1 are requested before tile t is issued, so no tile waits
    // on its table read
    auto read_id = [&](int t) {
      int id = -1;
      const int tok = t * kBn + lane * tpo;
      if (lane < a.ops_per_stage && tok < L) id = __ldg(a.block_tables + table_row + tok / a.block_size);
      return id;
    };
    int issued = 0;
    for (; issued < stop; ++issued) {
      const int slot = issued % LS;
      const int id_cur = id_next;
      if (issued + 1 < stop) id_next = read_id(issued + 1);
      if (issued >= LS &&
          !wait_or_abort(kv_empty(slot), ((issued / LS) - 1) & 1, abort, wait_ns)) {
        if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
        break;
      }
      const int t0 = issued * kBn;
      int blk = 0, off = 0;
      bool ok = false;
      if (lane < a.ops_per_stage) {
        const int t = t0 + lane * tpo;
        if (t < L) {
          const int j = t / a.block_size;
          off = t - j * a.block_size;
          blk = id_cur;
          ok = blk >= 0 && blk < a.num_blocks;
          if (!ok) atomicOr(a.err, PA_DEVERR_BLOCK_ID);
        }
      }
      const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) {
        uint64_t m = 0;
        for (int j = 0; j < a.ops_per_stage; ++j)
          if ((okmask >> j) & 1u) m |= ((tpo >= 64) ? ~0ull : ((1ull << tpo) - 1ull)) << (j * tpo);
        const int last = L - 1 - t0;  // tokens past the length hold no valid data
        if (last < kBn - 1) m &= (1ull << (last + 1)) - 1ull;
        masks[slot] = m;
        mbar_arrive_expect_tx(kv_full(slot),
                              static_cast<uint32_t>(__popc(okmask)) * tpo * kD * (FP8 ? 2u : 4u));
      }
      __syncwarp();
      if (ok) {
        if constexpr (FP8) {  // one 128-byte line of codes per token for K and for V
          const uint32_t dk = base + S::kCodes + slot * S::kCodeTile + lane * tpo * 128u;
          tma_load_4d(dk, &tmk, kv_full(slot), 0, kvh, off, blk);
          tma_load_4d(dk + S::kHalf, &tmv, kv_full(slot), 0, kvh, off, blk);
        } else {
          const uint32_t dk = base + S::kKRing + slot * S::kHalf + lane * tpo * 128u;
          const uint32_t dv = base + S::kVRing + slot * S::kHalf + lane * tpo * 128u;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            tma_load_4d(dk + c * S::kHalfStride, &tmk, kv_full(slot), c * 64, kvh, off, blk);
            tma_load_4d(dv + c * S::kHalfStride, &tmv, kv_full(slot), c * 64, kvh, off, blk);
          }
        }
      }
    }
    // copies in flight complete before the CTA frees its shared memory
    for (int j = (issued > LS ? issued - LS : 0); j < issued; ++j)
      mbar_wait_bounded(kv_full(j % LS), (j / LS) & 1, kLimitTcNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = umma_idesc(MB, kRowsTc, kBn, false);
    constexpr uint32_t id_o = umma_idesc(MB, kRowsTc, kD, true);
    // the tile the MMAs read: the ring stage itself, or (FP8) the widened buffer
    auto mma_tile = [&](int t) { return t % NB; };
    // wait until tile t is readable by the MMAs
    auto tile_ready = [&](int t) {
      return FP8 ? wait_or_abort(conv_full(t % NB), (t / NB) & 1, abort, wait_ns)
                 : wait_or_abort(kv_full(t % LS), (t / LS) & 1, abort, wait_ns);
    };
    // A descriptor's start address is its low 14 bits in 16-byte units and
    // shared memory stays below 256 KB, so an offset is a plain add: one
    // descriptor per operand and tile, then an add per MMA.
    const uint64_t dq0 = umma_desc(base + S::kQ, 16, 1024);
    auto issue_s = [&](int q, int t) {  // S_t of row tile q into its TMEM columns 64 * (t % 2)
      const uint64_t dq = dq0 + ((q * S::kQTile) >> 4);
      const uint64_t dk = umma_desc(base + S::kKRing + mma_tile(t) * S::kHalf, 16, 1024);
      const uint32_t d = tmem + q * 256u + (t & 1) * kBn;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (kRowsTc * 128u) + (kk & 3) * 32u;
        const uint32_t ko = (kk >> 2) * S::kHalfStride + (kk & 3) * 32u;
        umma(d, dq + (qo >> 4), dk + (ko >> 4), id_s, kk > 0 ? 1u : 0u);
      }
      umma_commit(s_full(q, t & 1));
    };
    auto issue_pv = [&](int q, int t) {  // O += P_t V_t of row tile q, P_t read from TMEM
      const uint64_t dv = umma_desc(base + S::kVRing + mma_tile(t) * S::kHalf, S::kHalfStride, 1024);
      const uint32_t p_col = tmem + q * 256u + (t & 1) * kBn;
      const uint32_t d = tmem + q * 256u + 2 * kBn;
#pragma unroll
      for (int part = 0; part < (MB ? 2 : 1); ++part) {
#pragma unroll
        for (int kk = 0; kk < kBn / 16; ++kk) {
          umma_tmem_a(d, p_col + part * (kBn / 2) + kk * 8u, dv + ((kk * 16u * 128u) >> 4), id_o,
                      (t > 0 || part > 0 || kk > 0) ? 1u : 0u);
        }
      }
      umma_commit(o_done(q, t & 1));
    };
    bool ok = true;
    if (lane == 0) {
      ok = tile_ready(0);
      if (ok) {
        tc_fence_after();
        for (int q = 0; q < kQTiles; ++q)
          if (nt[q] > 0) issue_s(q, 0);
      }
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles) {
          ok = tile_ready(t + 1);
          if (!ok) break;
          tc_fence_after();
          // S buffer (t+1) % 2 of a tile was released with its P_{t-1}
          for (int q = 0; q < kQTiles; ++q)
            if (t + 1 < nt[q]) issue_s(q, t + 1);
        }
        for (int q = 0; ok && q < kQTiles; ++q) {
          if (t >= nt[q]) continue;
          ok = wait_or_abort(p_full(q, t & 1), (t >> 1) & 1, abort, wait_ns);
          if (!ok) break;
          tc_fence_after();
          issue_pv(q, t);
        }
        if (ok) umma_commit(FP8 ? conv_empty(t % NB) : kv_empty(t % LS));
      }
      if (!ok) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
      umma_commit(fin);  // arrives once every MMA issued above has completed
      mbar_wait_bounded(fin, 0, kLimitTcNs);
    }
    __syncwarp();
  } else if (FP8 && warp >= kConvWarp) {
    // ------------------------------------------------------------ converters (FP8)
    // warp kConvWarp widens K, kConvWarp + 1 widens V (rows without valid data
    // become zeros). A code line of token t holds 8 chunks of 16 codes, chunk c
    // at (c ^ (t & 7)) * 16; its 32 fp16 bytes go to half c / 4, chunks
    // 2 (c % 4) and 2 (c % 4) + 1 of that token's line, swizzled the same way.
    const int which = warp - kConvWarp;  // 0: K, 1: V
    for (int t = 0; t < ntiles; ++t) {
      const int slot = t % LS;
      const int b = t % NB;
      if (!wait_or_abort(kv_full(slot), (t / LS) & 1, abort, wait_ns)) {
        if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
        break;
      }
      if (t >= NB && !wait_or_abort(conv_empty(b), ((t / NB) - 1) & 1, abort, wait_ns)) {
        if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
        break;
      }
      const uint64_t vmask = masks[slot];
      const uint32_t src = S::kCodes + slot * S::kCodeTile + which * S::kHalf;
      const uint32_t dst = (which ? S::kVRing : S::kKRing) + b * S::kHalf;
      // all of a batch's loads issue before its first store: the stores go to the
      // same shared array, so the compiler could not move a later load above them
      constexpr int kBatch = 8;
#pragma unroll
      for (int b0 = 0; b0 < kBn * 8 / 32; b0 += kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = (b0 + u) * 32 + lane;
          const int tok = idx >> 3;
          const int c = idx & 7;
          w[u] = *reinterpret_cast<const uint4*>(sm + src + tok * 128u + ((c ^ (tok & 7)) << 4));
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = (b0 + u) * 32 + lane;
          const int tok = idx >> 3;
          const int c = idx & 7;
          uint4 lo, hi;
          if (which == 1 && !((vmask >> tok) & 1ull)) {
            lo = hi = make_uint4(0u, 0u, 0u, 0u);
          } else {
            e4m3x4_to_f16(w[u].x, lo.x, lo.y);
            e4m3x4_to_f16(w[u].y, lo.z, lo.w);
            e4m3x4_to_f16(w[u].z, hi.x, hi.y);
            e4m3x4_to_f16(w[u].w, hi.z, hi.w);
          }
          const uint32_t line = dst + (c >> 2) * S::kHalfStride + tok * 128u;
          const int c2 = (c & 3) * 2;
          *reinterpret_cast<uint4*>(sm + line + ((c2 ^ (tok & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(sm + line + (((c2 + 1) ^ (tok & 7)) << 4)) = hi;
        }
      }
      if (which == 0 && lane == 0) conv_masks[b] = vmask;
      fence_proxy_async_smem();  // the MMAs read the widened tile through the async proxy
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(kv_empty(slot));  // the codes are no longer needed
        mbar_arrive(conv_full(b));
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int R = row0 + q * kRowsTc + r;
    const int i = R / g;
    const bool row_ok = R < rows;
    const int pos = row_ok ? L - n + i : -1;   // last key this row sees
    const uint32_t lane_base = tmem + q * 256u + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base;            // S buffers: + 64 * (t % 2)
    const uint32_t o_col = lane_base + 2 * kBn;  // O
    const float sl = a.scale_log2 * q_scale;
    const bool pos_scale = sl > 0.f;
    float m = -INFINITY;  // running max, log2 units
    float l = 0.f;
    bool ok = true;
    const int my_tiles = nt[q];
    for (int t = 0; t < my_tiles; ++t) {
      const int slot = t % LS;
      if (!wait_or_abort(s_full(q, t & 1), (t >> 1) & 1, abort, wait_ns)) { ok = false; break; }
      tc_fence_after();
      float x[kBn];
      tmem_ld64(s_col + (t & 1) * kBn, x);
      // the tile's valid-token mask: the producer wrote it before arming kv_full
      // (FP8: the K converter copied it before arming conv_full)
      uint64_t vmask;
      if constexpr (FP8) {
        if (!wait_or_abort(conv_full(t % NB), (t / NB) & 1, abort, wait_ns)) { ok = false; break; }
        vmask = conv_masks[t % NB];
      } else {
        if (!wait_or_abort(kv_full(slot), (t / LS) & 1, abort, wait_ns)) { ok = false; break; }
        vmask = masks[slot];
      }
      const int k0 = t * kBn;
      // logits in log2 units are x * sl; with sl > 0 the max commutes with the
      // scaling and the scaling folds into the exponent's FMA
      if (!pos_scale) {
#pragma unroll
        for (int c = 0; c < kBn; ++c) x[c] *= sl;
      }
      const float fs = pos_scale ? sl : 1.f;
      const bool whole = __all_sync(0xffffffffu, vmask == ~0ull && k0 + kBn - 1 <= pos);
      if (!whole) {
        const uint32_t mlo = static_cast<uint32_t>(vmask);
        const uint32_t mhi = static_cast<uint32_t>(vmask >> 32);
#pragma unroll
        for (int c = 0; c < kBn; ++c) {
          const bool valid = (k0 + c <= pos) && (((c < 32 ? mlo : mhi) >> (c & 31)) & 1u);
          x[c] = valid ? x[c] : -INFINITY;
        }
      }
      float mx;
      {  // 64 -> 22 -> 8 -> 3 -> 1 with three-input maxima
        float t22[22];
#pragma unroll
        for (int c = 0; c < 21; ++c) t22[c] = max3(x[c], x[c + 21], x[c + 42]);
        t22[21] = x[63];
        float t8[8];
#pragma unroll
        for (int c = 0; c < 7; ++c) t8[c] = max3(t22[c], t22[c + 7], t22[c + 14]);
        t8[7] = t22[21];
        mx = max3(max3(t8[0], t8[1], t8[2]), max3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7])) * fs;
      }
      const bool grow = mx > m + 8.f;
      const float m_new = grow ? mx : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = grow ? exp2f(m - m_use) : 1.f;
      // O is rescaled only after the previous O update of this tile completed
      if (t > 0 && __any_sync(0xffffffffu, grow && m != -INFINITY)) {
        if (!wait_or_abort(o_done(q, (t - 1) & 1), ((t - 1) >> 1) & 1, abort, wait_ns)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(o_col + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(o_col + c, o);
        }
      }
      m = m_new;
      uint32_t pk[kBn / 2];
      uint32_t pl[MB ? kBn / 2 : 1];
      uint64_t ps[kBn / 4];  // pair sums of p
      const uint64_t fs2 = f2(fs, fs);
      const uint64_t nm2 = f2(-m_use, -m_use);
#pragma unroll
      for (int c = 0; c < kBn; c += 2) {
        const float2 e = f2_split(fma_f2(f2(x[c], x[c + 1]), fs2, nm2));
        const float p0 = fast_exp2(e.x);
        const float p1 = fast_exp2(e.y);
        const uint64_t pp = f2(p0, p1);
        pk[c >> 1] = pack2<MB>(p0, p1);
        if constexpr (MB) {
          const float2 hi = unpack2<true>(pk[c >> 1]);
          const float2 lo = f2_split(sub_f2(pp, f2(hi.x, hi.y)));
          pl[c >> 1] = pack2<true>(lo.x, lo.y);
        }
        if ((c & 2) == 0) ps[c >> 2] = pp;
        else ps[c >> 2] = add_f2(ps[c >> 2], pp);
      }
#pragma unroll
      for (int w = kBn / 8; w >= 1; w >>= 1) {
#pragma unroll
        for (int c = 0; c < w; ++c) ps[c] = add_f2(ps[c], ps[c + w]);
      }
      const float2 psum = f2_split(ps[0]);
      l = l * alpha + (psum.x + psum.y);
      // P over this tile's S buffer: high part in its first 32 columns, low part next
      tmem_st32u(s_col + (t & 1) * kBn, pk);
      if constexpr (MB) tmem_st32u(s_col + (t & 1) * kBn + kBn / 2, pl);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // tokens without valid data: zero their V rows so 0 * garbage never
      // enters O (each row tile's warps zero the rows; the writes are equal).
      // FP8: the V converter wrote those rows as zeros.
      if (!FP8 && vmask != ~0ull) {
        const uint32_t vbase = S::kVRing + slot * S::kHalf;
        for (int idx = r; idx < kBn * 16; idx += kRowsTc) {
          const int tok = idx >> 4;
          const int rem = idx & 15;
          if (!((vmask >> tok) & 1ull))
            *reinterpret_cast<uint4*>(sm + vbase + (rem >> 3) * S::kHalfStride + tok * 128u + ((rem & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(q, t & 1));
    }
    if (!ok) {
      if (lane == 0) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
    } else if (my_tiles > 0) {
      // ---- epilogue: O / l once the last P V has completed
      if (wait_or_abort(o_done(q, (my_tiles - 1) & 1), ((my_tiles - 1) >> 1) & 1, abort, wait_ns)) {
        tc_fence_after();
        const float inv = l > 0.f ? (FP8 ? a.v_scale : 1.f) / l : 0.f;
        const int64_t ob = row_ok ? ((static_cast<int64_t>(q0) + i) * a.num_q_heads +
                                     static_cast<int64_t>(kvh) * g + R % g) * kD
                                  : 0;
#pragma unroll
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

template <bool IS_BF16, bool FP8>
cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a, dim3 grid,
                      cudaStream_t st) {
  auto kern = prefill_tc_e4m3_kernel<IS_BF16, FP8>;
  const int smem = static_cast<int>(TcSmem<FP8>::kTotal);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, tc_threads<FP8>(), smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc_e4m3(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const PrefillArgs& a, bool bf16, dim3 grid, cudaStream_t st) {
  return bf16 ? launch_tc<true, true>(tk, tv, a, grid, st) : launch_tc<false, true>(tk, tv, a, grid, st);
}

}  // namespace pa
