// pa_prefill_tc.cu - multi-token causal paged attention on the 5th-generation
// tensor cores (tcgen05 + TMEM) for head_dim 128.
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
// Masking: keys past a row's position get p = 0; V rows of tokens that hold no
// valid data (past the sequence's length, or of a block with an id out of
// range) are zeroed in shared memory before O += P V reads them. Every wait is
// bounded by %globaltimer; a CTA that gives up sets PA_DEVERR_TIMEOUT, drains
// what it has in flight (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kD = 128;            // head dim
constexpr int kRowsTc = 128;       // query rows per row tile (TMEM lanes)
constexpr int kQTiles = 2;         // row tiles per CTA
constexpr int kBn = 64;            // tokens per K/V tile
constexpr int kStagesTc = 4;       // K/V tiles in flight
constexpr int kSoftmaxWarps = 4 * kQTiles;
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
constexpr int kThreadsTc = (kSoftmaxWarps + 2) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kLimitTcNs = 2000000000ull;

struct TcSmem {
  static constexpr uint32_t kHalf = kBn * 128;                  // 64 token rows of 128 bytes
  static constexpr uint32_t kQTile = 2 * kRowsTc * 128;         // 2 halves x 128 rows x 128 B
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kStage = 4 * kHalf;                 // K halves, then V halves
  static constexpr uint32_t kStages = kQ + kQTiles * kQTile;
  static constexpr uint32_t kBar = kStages + kStagesTc * kStage;
  // kv_full[NS], kv_empty[NS], s_full[2 tiles][2], p_full[2 tiles][2],
  // o_done[2 tiles][2], final. p_full and o_done alternate by tile parity: a
  // softmax warp may publish P_{t+1} before the MMA warp waits for P_t, and
  // waits on o_done only now and then, so a single barrier could run two
  // phases ahead of its waiter, where parity waits alias.
  static constexpr uint32_t kNumBars = 2 * kStagesTc + 4 + 4 + 4 + 1;
  static constexpr uint32_t kMask = kBar + kNumBars * 8;        // uint64 per stage
  static constexpr uint32_t kMisc = kMask + kStagesTc * 8;      // tmem base, abort flag
  static constexpr uint32_t kTotal = kMisc + 16 + 1024;         // + base-alignment slack
};
static_assert(TcSmem::kTotal <= 232448, "shared memory budget");

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, A/B fp16 or bf16, M x N,
// A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t umma_idesc(bool bf16, int m, int n, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// The same with the A operand in tensor memory (row m in lane m, 16-bit pairs
// per 32-bit column).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 TMEM columns of this thread's lane: two loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
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
#undef PA_LD32
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x on the SFU (ex2.approx, flushing subnormal results to zero); the softmax
// arguments are at most 8.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 packed 32-bit words into consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns` while
// the phase is incomplete, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait that also gives up once another role of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (*abort != 0u || globaltimer_ns() - t0 > kLimitTcNs) return false;
  }
  return true;
}

// Grid: (row-pair tiles, H_kv, N); x is taken in reverse so the tiles with the
// largest positions (most K/V) start first.
template <bool IS_BF16>
__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using S = TcSmem;
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
  uint64_t* masks = reinterpret_cast<uint64_t*>(sm + S::kMask);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kMisc);
  volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(sm + S::kMisc + 4);

  if (threadIdx.x == 0) {
    for (int k = 0; k < kStagesTc; ++k) {
      mbar_init(kv_full(k), 1);
      mbar_init(kv_empty(k), 1);
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

  // ---- Q rows into shared memory (K-major, 128-byte swizzle), one row per thread
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
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = src != nullptr ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t off = S::kQ + q * S::kQTile + (c >> 3) * (kRowsTc * 128u) + r * 128u +
                           (((c & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sm + off) = v;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t table_row = static_cast<int64_t>(s) * a.max_blocks;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    const int tpo = a.tok_per_op;
    int issued = 0;
    for (; issued < ntiles; ++issued) {
      const int slot = issued % kStagesTc;
      if (issued >= kStagesTc &&
          !wait_or_abort(kv_empty(slot), ((issued / kStagesTc) - 1) & 1, abort)) {
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
          blk = __ldg(a.block_tables + table_row + j);
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
        mbar_arrive_expect_tx(kv_full(slot), static_cast<uint32_t>(__popc(okmask)) * tpo * kD * 4u);
      }
      __syncwarp();
      if (ok) {
        const uint32_t dk = base + S::kStages + slot * S::kStage + lane * tpo * 128u;
        const uint32_t dv = dk + 2 * S::kHalf;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tma_load_4d(dk + c * S::kHalf, &tmk, kv_full(slot), c * 64, kvh, off, blk);
          tma_load_4d(dv + c * S::kHalf, &tmv, kv_full(slot), c * 64, kvh, off, blk);
        }
      }
    }
    // copies in flight complete before the CTA frees its shared memory
    for (int j = (issued > kStagesTc ? issued - kStagesTc : 0); j < issued; ++j)
      mbar_wait_bounded(kv_full(j % kStagesTc), (j / kStagesTc) & 1, kLimitTcNs);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = umma_idesc(IS_BF16, kRowsTc, kBn, false);
    constexpr uint32_t id_o = umma_idesc(IS_BF16, kRowsTc, kD, true);
    auto issue_s = [&](int q, int t) {  // S_t of row tile q into its TMEM columns 64 * (t % 2)
      const uint32_t q_addr = base + S::kQ + q * S::kQTile;
      const uint32_t k_addr = base + S::kStages + (t % kStagesTc) * S::kStage;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t qo = (kk >> 2) * (kRowsTc * 128u) + (kk & 3) * 32u;
        const uint32_t ko = (kk >> 2) * S::kHalf + (kk & 3) * 32u;
        umma(tmem + q * 256u + (t & 1) * kBn, umma_desc(q_addr + qo, 16, 1024),
             umma_desc(k_addr + ko, 16, 1024), id_s, kk > 0 ? 1u : 0u);
      }
      umma_commit(s_full(q, t & 1));
    };
    auto issue_pv = [&](int q, int t) {  // O += P_t V_t of row tile q, P_t read from TMEM
      const uint32_t v_addr = base + S::kStages + (t % kStagesTc) * S::kStage + 2 * S::kHalf;
      const uint32_t p_col = tmem + q * 256u + (t & 1) * kBn;
#pragma unroll
      for (int part = 0; part < (IS_BF16 ? 2 : 1); ++part) {
#pragma unroll
        for (int kk = 0; kk < kBn / 16; ++kk) {
          umma_tmem_a(tmem + q * 256u + 2 * kBn, p_col + part * (kBn / 2) + kk * 8u,
                      umma_desc(v_addr + kk * 16u * 128u, S::kHalf, 1024), id_o,
                      (t > 0 || part > 0 || kk > 0) ? 1u : 0u);
        }
      }
      umma_commit(o_done(q, t & 1));
    };
    bool ok = true;
    if (lane == 0) {
      ok = wait_or_abort(kv_full(0), 0, abort);
      if (ok) {
        tc_fence_after();
        for (int q = 0; q < kQTiles; ++q)
          if (nt[q] > 0) issue_s(q, 0);
      }
      for (int t = 0; ok && t < ntiles; ++t) {
        if (t + 1 < ntiles) {
          ok = wait_or_abort(kv_full((t + 1) % kStagesTc), ((t + 1) / kStagesTc) & 1, abort);
          if (!ok) break;
          tc_fence_after();
          // S buffer (t+1) % 2 of a tile was released with its P_{t-1}
          for (int q = 0; q < kQTiles; ++q)
            if (t + 1 < nt[q]) issue_s(q, t + 1);
        }
        for (int q = 0; ok && q < kQTiles; ++q) {
          if (t >= nt[q]) continue;
          ok = wait_or_abort(p_full(q, t & 1), (t >> 1) & 1, abort);
          if (!ok) break;
          tc_fence_after();
          issue_pv(q, t);
        }
        if (ok) umma_commit(kv_empty(t % kStagesTc));
      }
      if (!ok) { atomicOr(a.err, PA_DEVERR_TIMEOUT); *abort = 1u; }
      umma_commit(fin);  // arrives once every MMA issued above has completed
      mbar_wait_bounded(fin, 0, kLimitTcNs);
    }
    __syncwarp();
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
    const float sl = a.scale_log2;
    const bool pos_scale = sl > 0.f;
    float m = -INFINITY;  // running max, log2 units
    float l = 0.f;
    bool ok = true;
    const int my_tiles = nt[q];
    for (int t = 0; t < my_tiles; ++t) {
      const int slot = t % kStagesTc;
      if (!wait_or_abort(s_full(q, t & 1), (t >> 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      float x[kBn];
      tmem_ld64(s_col + (t & 1) * kBn, x);
      // the tile's valid-token mask: the producer wrote it before arming kv_full
      if (!wait_or_abort(kv_full(slot), (t / kStagesTc) & 1, abort)) { ok = false; break; }
      const uint64_t vmask = masks[slot];
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
      {
        float t32[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) t32[c] = fmaxf(x[c], x[c + 32]);
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
          for (int c = 0; c < w; ++c) t32[c] = fmaxf(t32[c], t32[c + w]);
        }
        mx = t32[0] * fs;
      }
      const bool grow = mx > m + 8.f;
      const float m_new = grow ? mx : m;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = grow ? exp2f(m - m_use) : 1.f;
      // O is rescaled only after the previous O update of this tile completed
      if (t > 0 && __any_sync(0xffffffffu, grow && m != -INFINITY)) {
        if (!wait_or_abort(o_done(q, (t - 1) & 1), ((t - 1) >> 1) & 1, abort)) { ok = false; break; }
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
      uint32_t pl[IS_BF16 ? kBn / 2 : 1];
      float ps[kBn / 2];
#pragma unroll
      for (int c = 0; c < kBn; c += 2) {
        const float p0 = fast_exp2(fmaf(x[c], fs, -m_use));
        const float p1 = fast_exp2(fmaf(x[c + 1], fs, -m_use));
        pk[c >> 1] = pack2<IS_BF16>(p0, p1);
        if constexpr (IS_BF16) {
          const float2 hi = unpack2<true>(pk[c >> 1]);
          pl[c >> 1] = pack2<true>(p0 - hi.x, p1 - hi.y);
        }
        ps[c >> 1] = p0 + p1;
      }
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
        for (int c = 0; c < w; ++c) ps[c] += ps[c + w];
      }
      l = l * alpha + ps[0];
      // P over this tile's S buffer: high part in its first 32 columns, low part next
      tmem_st32u(s_col + (t & 1) * kBn, pk);
      if constexpr (IS_BF16) tmem_st32u(s_col + (t & 1) * kBn + kBn / 2, pl);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // tokens without valid data: zero their V rows so 0 * garbage never
      // enters O (each row tile's warps zero the rows; the writes are equal)
      if (vmask != ~0ull) {
        const uint32_t vbase = S::kStages + slot * S::kStage + 2 * S::kHalf;
        for (int idx = r; idx < kBn * 16; idx += kRowsTc) {
          const int tok = idx >> 4;
          const int rem = idx & 15;
          if (!((vmask >> tok) & 1ull))
            *reinterpret_cast<uint4*>(sm + vbase + (rem >> 3) * S::kHalf + tok * 128u + ((rem & 7) << 4)) =
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
      if (wait_or_abort(o_done(q, (my_tiles - 1) & 1), ((my_tiles - 1) >> 1) & 1, abort)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
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

template <bool IS_BF16>
cudaError_t launch_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a, dim3 grid,
                      cudaStream_t st) {
  auto kern = prefill_tc_kernel<IS_BF16>;
  const int smem = static_cast<int>(TcSmem::kTotal);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreadsTc, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                              bool bf16, dim3 grid, cudaStream_t st) {
  return bf16 ? launch_tc<true>(tk, tv, a, grid, st) : launch_tc<false>(tk, tv, a, grid, st);
}

}  // namespace pa
