// pa_prefix_hash.cu - prefix-cache keys of full blocks, computed on the device.
//
// A cached block is found again by its content: a hit needs an unbroken chain
// of matching block keys from position zero, and the first differing token
// ends the chain ("Paged Attention", firehose-demo; "PagedAttention",
// learn.pranaymahendrakar.com, Prefix caching: hash each block-aligned prefix
// of token ids). Each full block j of a sequence gets
//   key_j = SHA-256(key_{j-1} || token ids of block j as int32 little-endian),
// key_{-1} = a 32-byte root; a trailing partial block gets no key.
//
// SHA-256 follows FIPS 180-4: message padded with one 1 bit, zeros and the
// 64-bit big-endian bit length to whole 64-byte chunks; each chunk expands to
// 64 schedule words and runs 64 rounds over eight 32-bit state words. The
// round constants and the initial state are, by the standard's definition, the
// first 32 fraction bits of the cube roots of the first 64 primes and of the
// square roots of the first 8; they are derived here on the host with exact
// integer roots at first use and passed to the kernel as parameters.
//
// The chain is sequential within a sequence, so one thread walks one
// sequence; sequences run in parallel. The parent key (8 words) and the block's
// ids are the message words in order, so chunk 0 always starts with the
// parent and no state is ever indexed at run time.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {

namespace {

uint64_t icbrt(unsigned __int128 n) {  // floor(n^(1/3)), n < 2^120
  uint64_t lo = 0, hi = 1ull << 40;
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo + 1) / 2;
    const unsigned __int128 m = mid;
    if (m * m * m <= n) lo = mid; else hi = mid - 1;
  }
  return lo;
}

uint64_t isqrt(unsigned __int128 n) {  // floor(n^(1/2)), n < 2^80
  uint64_t lo = 0, hi = 1ull << 40;
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo + 1) / 2;
    const unsigned __int128 m = mid;
    if (m * m <= n) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace

const Sha256Consts& sha256_consts() {
  static Sha256Consts c;
  static std::once_flag once;
  std::call_once(once, [] {
    uint32_t primes[64];
    int n = 0;
    for (uint32_t p = 2; n < 64; ++p) {
      bool prime = true;
      for (uint32_t q = 2; q * q <= p; ++q)
        if (p % q == 0) { prime = false; break; }
      if (prime) primes[n++] = p;
    }
    for (int i = 0; i < 64; ++i)  // floor(cbrt(p) * 2^32) mod 2^32
      c.k[i] = static_cast<uint32_t>(icbrt(static_cast<unsigned __int128>(primes[i]) << 96));
    for (int i = 0; i < 8; ++i)   // floor(sqrt(p) * 2^32) mod 2^32
      c.h0[i] = static_cast<uint32_t>(isqrt(static_cast<unsigned __int128>(primes[i]) << 64));
  });
  return c;
}

namespace {

__device__ __forceinline__ uint32_t rotr(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

// One SHA-256 compression of the 16 message words w into state st.
__device__ __forceinline__ void sha256_compress(uint32_t (&st)[8], uint32_t (&w)[16],
                                                const Sha256Consts& c) {
  uint32_t a = st[0], b = st[1], cc = st[2], d = st[3], e = st[4], f = st[5], g = st[6], h = st[7];
#pragma unroll
  for (int t = 0; t < 64; ++t) {
    uint32_t wt;
    if (t < 16) {
      wt = w[t];
    } else {
      const uint32_t w15 = w[(t - 15) & 15];
      const uint32_t w2 = w[(t - 2) & 15];
      const uint32_t s0 = rotr(w15, 7) ^ rotr(w15, 18) ^ (w15 >> 3);
      const uint32_t s1 = rotr(w2, 17) ^ rotr(w2, 19) ^ (w2 >> 10);
      wt = w[t & 15] + s0 + w[(t - 7) & 15] + s1;
      w[t & 15] = wt;
    }
    const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = h + S1 + ch + c.k[t] + wt;
    const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & b) ^ (a & cc) ^ (b & cc);
    const uint32_t t2 = S0 + maj;
    h = g;
    g = f;
    f = e;
    e = d + t1;
    d = cc;
    cc = b;
    b = a;
    a = t1 + t2;
  }
  st[0] += a; st[1] += b; st[2] += cc; st[3] += d;
  st[4] += e; st[5] += f; st[6] += g; st[7] += h;
}

__global__ void prefix_hash_kernel(const int32_t* __restrict__ tokens,
                                   const int64_t* __restrict__ tok_off,
                                   const int64_t* __restrict__ key_off, int32_t num_seqs,
                                   int32_t block_size, const Sha256Consts c, const Sha256Root root,
                                   uint32_t* __restrict__ keys, int* err) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= num_seqs) return;
  const int64_t t0 = tok_off[s];
  const int64_t n = tok_off[s + 1] - t0;
  const int64_t k0 = key_off[s];
  if (n < 0 || key_off[s + 1] - k0 != n / block_size) {
    atomicOr(err, PA_DEVERR_SEQ_LEN);
    return;
  }
  const int64_t nk = n / block_size;
  // message: 8 parent words, block_size token words, 0x80000000, zeros, 2 length words
  const int words = 8 + block_size;
  const int total = ((words + 1 + 2 + 15) / 16) * 16;
  const uint64_t bits = static_cast<uint64_t>(words) * 32u;
  uint32_t parent[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) parent[i] = root.w[i];
  for (int64_t j = 0; j < nk; ++j) {
    const int32_t* blk = tokens + t0 + j * block_size;
    uint32_t st[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) st[i] = c.h0[i];
    for (int ch = 0; ch < total / 16; ++ch) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int idx = ch * 16 + i;
        uint32_t v;
        if (i < 8 && ch == 0) {
          v = parent[i];
        } else if (idx < words) {
          v = __byte_perm(static_cast<uint32_t>(__ldg(blk + (idx - 8))), 0u, 0x0123);  // LE bytes
        } else if (idx == words) {
          v = 0x80000000u;
        } else if (idx == total - 2) {
          v = static_cast<uint32_t>(bits >> 32);
        } else if (idx == total - 1) {
          v = static_cast<uint32_t>(bits);
        } else {
          v = 0u;
        }
        w[i] = v;
      }
      sha256_compress(st, w, c);
    }
    uint32_t* out = keys + (k0 + j) * 8;
    // the digest's bytes are the state words big-endian; store them byte-swapped
    // so memory holds that byte order
    uint4 lo, hi;
    lo.x = __byte_perm(st[0], 0u, 0x0123); lo.y = __byte_perm(st[1], 0u, 0x0123);
    lo.z = __byte_perm(st[2], 0u, 0x0123); lo.w = __byte_perm(st[3], 0u, 0x0123);
    hi.x = __byte_perm(st[4], 0u, 0x0123); hi.y = __byte_perm(st[5], 0u, 0x0123);
    hi.z = __byte_perm(st[6], 0u, 0x0123); hi.w = __byte_perm(st[7], 0u, 0x0123);
    reinterpret_cast<uint4*>(out)[0] = lo;
    reinterpret_cast<uint4*>(out)[1] = hi;
#pragma unroll
    for (int i = 0; i < 8; ++i) parent[i] = st[i];
  }
}

// key_off[0] = 0, key_off[s + 1] = key_off[s] + floor(len_s / block_size):
// the first key of each sequence when keys are packed back to back. One CTA
// scans chunks of kScanThreads * kScanItems sequences in order, each thread
// summing kScanItems consecutive counts before a block-wide exclusive scan of
// the thread totals; the running carry moves on to the next chunk. A negative
// length counts as zero keys and sets PA_DEVERR_SEQ_LEN (the hash kernel then
// skips that sequence).
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 8;

__global__ void __launch_bounds__(kScanThreads)
    key_offsets_kernel(const int64_t* __restrict__ tok_off, int32_t num_seqs, int32_t block_size,
                       int64_t* __restrict__ key_off, int* err) {
  __shared__ int64_t warp_sums[kScanThreads / 32];
  __shared__ int64_t carry_s;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    carry_s = 0;
    key_off[0] = 0;
  }
  __syncthreads();
  constexpr int kChunk = kScanThreads * kScanItems;
  for (int64_t base = 0; base < num_seqs; base += kChunk) {
    const int64_t s0 = base + static_cast<int64_t>(threadIdx.x) * kScanItems;
    int64_t cnt[kScanItems];
    int64_t mine = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      const int64_t s = s0 + i;
      int64_t c = 0;
      if (s < num_seqs) {
        const int64_t n = tok_off[s + 1] - tok_off[s];
        if (n < 0) bad = true;
        c = n > 0 ? n / block_size : 0;
      }
      cnt[i] = c;
      mine += c;
    }
    if (bad) atomicOr(err, PA_DEVERR_SEQ_LEN);
    // inclusive scan of the thread totals: within each warp, then across warps
    int64_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int64_t w = warp_sums[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t carry = carry_s;
    int64_t run = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - mine;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      const int64_t s = s0 + i;
      run += cnt[i];
      if (s < num_seqs) key_off[s + 1] = run;
    }
    __syncthreads();  // every thread has read carry_s and warp_sums
    if (threadIdx.x == 0) carry_s = carry + warp_sums[kScanThreads / 32 - 1];
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_key_offsets(const int64_t* tok_off, int32_t num_seqs, int32_t block_size,
                               int64_t* key_off, int* err, cudaStream_t st) {
  key_offsets_kernel<<<1, kScanThreads, 0, st>>>(tok_off, num_seqs, block_size, key_off, err);
  return cudaGetLastError();
}

cudaError_t launch_prefix_hash(const int32_t* tokens, const int64_t* tok_off, const int64_t* key_off,
                               int32_t num_seqs, int32_t block_size, const Sha256Root& root,
                               uint8_t* keys, int* err, cudaStream_t st) {
  const int threads = 64;
  const int blocks = (num_seqs + threads - 1) / threads;
  prefix_hash_kernel<<<blocks, threads, 0, st>>>(tokens, tok_off, key_off, num_seqs, block_size,
                                                 sha256_consts(), root,
                                                 reinterpret_cast<uint32_t*>(keys), err);
  return cudaGetLastError();
}

}  // namespace pa
