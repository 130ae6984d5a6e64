// pa_chunk_umma.cuh -- paged attention for chunks of query tokens on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// What it computes is pa_attention_varlen's definition ("Inside vLLM CUDA Kernels",
// Part 3, FlashAttention over paged KV: a CTA owns a Q tile, resolves and loads the K/V
// tiles of its sequence through block_table while scanning the K dimension, and runs
// QK, online softmax and P.V on each): query i of a sequence with n new tokens sits at
// position len - n + i and sees the tokens up to it; the logit is scale q.k (+ the ALiBi
// bias slope_h (t - position)).
//
// Work unit (one CTA): sequence s, KV head g and one or two tiles of 128 query rows --
// row r of the KV head is query token r / G at head g G + r % G.  The page range is scanned in groups of 4
// pages (64 tokens):
//   S[128 x 64] = Q[128 x D] . K_group^T        tcgen05.mma, A and B from shared memory,
//                                               S in tensor memory (TMEM)
//   softmax, one thread per row                 tcgen05.ld of the row's 64 scores; lazy
//                                               running max; P written back over S as
//                                               16-bit hi + lo halves (tcgen05.st)
//   O[128 x D] += P[128 x 16] . V_page[16 x D]  tcgen05.mma per page and half, A = P from
//                                               TMEM, B = the V page in shared memory
// Roles (T tiles): warps 0 .. 4T-1 run the softmax and the epilogue (warp w belongs to
// tile w / 4 and owns its TMEM lanes and rows 32 (w % 4) ..); warp 4T + t issues the MMAs
// of tile t (the whole warp runs the loop, one elected lane issues), warp 4T also allocates
// TMEM; warp 5T resolves block_table and issues the TMA page loads into a ring of R page
// slots.
// Shared memory holds Q (loaded by the softmax threads, 128-byte swizzle) and the K and V
// rings, one region per 64-element box of a row, so that the 16-token pages of a group
// sit at one 1024-byte stride per 8 rows and form one MMA operand.  S and P of groups k
// and k + 1 use two TMEM buffers; O lives in TMEM until the epilogue normalises it.
//
// Synchronisation (mbarriers, every wait bounded and abandoned when another role gave
// up): full[slot] (TMA bytes) -> the issuers; per tile s_full[b] (commit) -> softmax,
// p_full[b] (128 arrivals) -> its issuer, o_done (commit after each group's P.V) ->
// softmax, only before an O rescale and the epilogue (S of group k is issued after P.V of
// group k - 2, so its completion bounds o_done's phase from below and a parity wait cannot
// be a phase off); empty[slot] (one commit per active tile) -> TMA.  The MMAs
// of one issuer run in order, so S of group k + 2 may overwrite the P that P.V of group k
// reads.  Tile 0 zeroes the V rows past the sequence in the last page before it hands over
// its P and arrives on v_tail (used once), which the other tiles' last P.V waits for.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_merge.cuh"  // grid_dependency_wait

namespace pa {

namespace umma {

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (TMEM) (+)= A (shared memory descriptor) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D (TMEM) (+)= A (TMEM) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// One arrival on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane; the wait is in the same
// statement so that no use of the values can be scheduled before it.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 consecutive columns as two 32-column loads under one wait.
__device__ __forceinline__ void ld32x2(uint32_t taddr, float (&v)[32], float (&w)[32]) {
  uint32_t r[32], q[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, "
      "%46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]),
        "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15]),
        "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]),
        "=r"(q[24]), "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(r[i]);
    w[i] = __uint_as_float(q[i]);
  }
}
__device__ __forceinline__ void st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared memory matrix descriptor: 128-byte swizzle, start address, leading and stride
// byte offsets (16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: f32 accumulator, A and B both bf16 (or both f16),
// A K-major, B K-major or MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc(bool bf, bool b_mn_major, int M, int N) {
  return (1u << 4) | ((bf ? 1u : 0u) << 7) | ((bf ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace umma

// Packed fp32 pairs (one 64-bit register pair, low half first) and the two-lane
// round-to-nearest arithmetic on them; a three-input max.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

constexpr uint32_t kUmmaWaitLimit = 1u << 20;  // mbarrier polls before a wait gives up
constexpr float kUmmaSlack = 8.f;              // lazy running max, log2 units (p <= 256)
constexpr float kUmmaEmpty = -1e30f;           // running max of a row with no visible token yet

// T row tiles of 128 rows per CTA.  T = 1: 6 warps, two CTAs per SM (their softmax and
// MMA phases interleave).  T = 2: 10 warps, one CTA per SM; both tiles consume every K/V
// page that is loaded once, and the ring is deeper.
template <int KIND, int D, int T>
struct UmmaCfg {
  static constexpr bool BF = KIND == KIND_BF16;
  static constexpr int TILES = T, ROWS = 128 * T;
  // warps 0 .. 4T-1 softmax, 4T .. 5T-1 one MMA issuer per tile, 5T the TMA producer
  static constexpr int MMA_WARP = 4 * T, TMA_WARP = 5 * T, THREADS = (5 * T + 1) * 32;
  static constexpr int MIN_CTAS = T == 1 ? 2 : 1;
  static constexpr int NBOX = D / 64;                 // 64-element (128-byte) boxes per row
  static constexpr int GP = 4;                        // pages per group: 64 tokens
  static constexpr int R = T == 1 ? (D == 64 ? 16 : 8) : (D == 64 ? 40 : 20);  // page slots of the ring
  static constexpr int NS = R / GP;                   // group slots
  static constexpr int BOXB = kBlock * 128;           // one page's rows of one box: 2 KiB
  static constexpr int QBOX = 128 * 128;              // one box of one 128-row Q tile: 16 KiB
  static constexpr int QTILE = NBOX * QBOX;           // one Q tile
  static constexpr int RING = R * BOXB;               // one box region of a ring
  static constexpr int QOFF = 0, KOFF = T * QTILE, VOFF = KOFF + NBOX * RING, BAR_OFF = VOFF + NBOX * RING;
  // barriers: full[NS], empty[NS]; per tile s_full x2, p_full x2, o_done, drain (48 bytes);
  // q_full, v_tail
  static constexpr int TBAR = 2 * NS * 8, NBARS = 2 * NS + 6 * T + 2;
  static constexpr size_t SMEM = 1024 + BAR_OFF + NBARS * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 256 * T;      // tile t: S/P buffers at 256 t + 0 / 64, O at 256 t + 128
  static constexpr uint32_t OCOL = 128;
  static_assert(D % 64 == 0 && D <= 128, "head size 64 or 128");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Bounded mbarrier wait that also gives up once another role has set *abort.
__device__ __forceinline__ bool umma_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint32_t limit = kUmmaWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

template <int KIND, int D, int T>
__global__ void __launch_bounds__(UmmaCfg<KIND, D, T>::THREADS, UmmaCfg<KIND, D, T>::MIN_CTAS)
    chunk_umma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ) {
  using C = UmmaCfg<KIND, D, T>;
  using OutT = typename std::conditional<C::BF, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KiB alignment
  uint8_t *sgen = smem_raw + (sbase - raw_u32);
  const uint32_t qs = sbase + C::QOFF, ks = sbase + C::KOFF, vs = sbase + C::VOFF;
  const uint32_t full0 = sbase + C::BAR_OFF, empty0 = full0 + 8 * C::NS, tbar0 = full0 + C::TBAR;
  // barriers of tile t
  auto sfull = [&](int t, int b) { return tbar0 + 48u * t + 8u * b; };
  auto pfull = [&](int t, int b) { return tbar0 + 48u * t + 16u + 8u * b; };
  auto odone = [&](int t) { return tbar0 + 48u * t + 32u; };
  auto drain = [&](int t) { return tbar0 + 48u * t + 40u; };
  const uint32_t qfull = tbar0 + 48u * T, vtailb = qfull + 8u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sgen + C::BAR_OFF + C::NBARS * 8);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *bad_block = reinterpret_cast<volatile int *>(tmem_slot + 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rt = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int G = p.G;

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    if (p.q_tma) prefetch_tensormap(&tmQ);
  }
  grid_dependency_wait();

  const int len = __ldg(p.seq_lens + s);
  const int a = __ldg(p.qsl + s), b_end = __ldg(p.qsl + s + 1);
  const int nq = b_end - a;
  if (len < 0 || len > p.max_blocks * kBlock || a < 0 || b_end > p.Tq || nq < 0 || nq > p.nq_max || nq > len) {
    if (tid == 0 && rt == 0 && g == 0 && p.err) atomicOr(p.err, kErrSeqLen);
    return;
  }
  const int r0 = rt * C::ROWS;                  // first row of the CTA
  const int nrows = min(C::ROWS, nq * G - r0);  // rows with a query token
  if (nrows <= 0) return;
  const int ntiles = (nrows + 127) / 128;       // tiles with a query row
  const int pos0 = len - nq;                    // row r sees tokens 0 .. pos0 + r / G
  const int vis = pos0 + (r0 + nrows - 1) / G + 1;
  const int npages = (vis + kBlock - 1) / kBlock;
  const int ngr = (npages + C::GP - 1) / C::GP;
  if (tid == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, ntiles);  // one commit per active tile's issuer
    }
    for (int t = 0; t < T; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(sfull(t, b), 1);
        mbar_init(pfull(t, b), 128);
      }
      mbar_init(odone(t), 1);
      mbar_init(drain(t), 1);
    }
    mbar_init(qfull, 1);
    mbar_init(vtailb, 128);
    *abort = 0;
    *bad_block = 0;
    fence_barrier_init();
  }
  // The barriers are initialised: the TMA producer starts on Q and the first K/V pages now,
  // the other roles meet again below once TMEM is allocated (and Q is stored, without TMA).
  __syncthreads();

  // ---- Q tiles -> shared memory by the softmax threads when there is no Q tensor map:
  // the 128-byte swizzle TMA gives, zero rows past nrows
  if (!p.q_tma && tid < C::ROWS) {
    const int r = r0 + tid, tr = tid & 127;
    const bool valid = tid < nrows;
    const uint4 *src = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(p.q) +
        ((static_cast<int64_t>(a) + r / G) * p.q_ss + static_cast<int64_t>(g * G + r % G) * p.q_hs) * 2);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const int box = c >> 3, ch = c & 7;
      *reinterpret_cast<uint4 *>(sgen + C::QOFF + (tid >> 7) * C::QTILE + box * C::QBOX + (tr >> 3) * 1024 +
                                 (tr & 7) * 128 + ((ch ^ (tr & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();  // generic writes -> the tensor core's async reads
  }
  if (warp == C::MMA_WARP) {
    umma::tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    umma::tmem_relinquish();
  }
  if (warp != C::TMA_WARP) {
    // every role but the producer: the TMEM address and a Q the threads stored (named barrier 1)
    umma::fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(C::THREADS - 32) : "memory");
    umma::fence_after();
  }
  const uint32_t tmem = warp == C::TMA_WARP ? 0u : *reinterpret_cast<volatile uint32_t *>(tmem_slot);

  // softmax state of row r0 + tid (threads below ROWS: tile tid / 128), kept for the epilogue
  const int row = r0 + tid;
  const bool valid = tid < nrows;
  const int tile = warp >> 2;
  // the warp's TMEM lanes (a warp reaches lanes 32 (warp % 4) ..) in its tile's columns
  const uint32_t tl = tmem + 256u * tile + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  float l = 0.f;
  bool ok = true;
  int issued = 0;  // TMA producer: K/V groups issued

  if (warp == C::TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    const int32_t *bt = p.block_table + static_cast<int64_t>(s) * p.bt_ss;
    const uint64_t pol = policy_evict_normal();  // the other row tiles of (s, g) read the same pages
    const int c1 = p.nhd ? g : 0, c2 = p.nhd ? 0 : g;
    // block-table entries are read one group ahead, off the path from a free slot to its copies
    int pid_next = lane < min(C::GP, npages) ? __ldg(bt + lane) : 0;
    if (p.q_tma && lane == 0) {
      // Q first: the row tiles' boxes (query tokens x G heads x 64 dims each); rows past nrows
      // hold other tokens or zeros, and only feed rows that are never stored
      mbar_arrive_expect_tx(qfull, ntiles * C::NBOX * C::QBOX);
      const uint64_t qpol = policy_evict_first();
      for (int t = 0; t < ntiles; ++t)
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx)
          tma_load_3d(qs + t * C::QTILE + bx * C::QBOX, &tmQ, qfull, bx * 64, g * G, a + (r0 + 128 * t) / G, qpol);
    }
    for (int k = 0; k < ngr; ++k) {
      const int gs = k % C::NS;
      if (k >= C::NS && !__all_sync(0xffffffffu, umma_wait(empty0 + 8 * gs, ((k / C::NS) - 1) & 1, abort))) break;
      const int npg = min(C::GP, npages - k * C::GP);
      int pid = pid_next;
      if (k + 1 < ngr) pid_next = lane < min(C::GP, npages - (k + 1) * C::GP) ? __ldg(bt + (k + 1) * C::GP + lane) : 0;
      if (lane < npg && (pid < 0 || pid >= p.num_blocks)) {
        *bad_block = 1;
        if (p.err) atomicOr(p.err, kErrBlock);
        pid = 0;  // load a valid block; the CTA writes nothing
      }
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * gs, npg * 2 * C::NBOX * C::BOXB);
      __syncwarp();
      if (lane < npg) {
        const int slot = gs * C::GP + lane;
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
          tma_load_4d(ks + bx * C::RING + slot * C::BOXB, &tmK, full0 + 8 * gs, bx * 64, c1, c2, pid, pol);
          tma_load_4d(vs + bx * C::RING + slot * C::BOXB, &tmV, full0 + 8 * gs, bx * 64, c1, c2, pid, pol);
        }
      }
      issued = k + 1;
    }
  } else if (warp >= C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer of tile t
    // The whole warp runs the loop, so descriptors and addresses are warp-uniform values;
    // one elected lane issues each batch of MMAs and its commit.  Each tile has its own
    // issuer, so a tile whose softmax runs late does not hold back the other.
    const int t = warp - C::MMA_WARP;
    if (t < ntiles) {
      constexpr uint32_t iS = umma::idesc(C::BF, false, 128, 64);  // S = Q . K^T, N = 64 tokens
      constexpr uint32_t iPV = umma::idesc(C::BF, true, 128, D);   // O += P . V, N = D dims
      // descriptors are built once; an operand at a byte offset adds offset / 16 to them
      const uint64_t qd = umma::sdesc(qs + t * C::QTILE, 16, 1024), kd0 = umma::sdesc(ks, 16, 1024);
      // V (MN-major): 8-token row groups 1024 bytes apart, the 64-dim boxes one ring region apart
      const uint64_t vd0 = umma::sdesc(vs, C::RING, 1024);
      const uint32_t tt = tmem + 256u * t;  // the tile's TMEM columns
      const bool vtail = len - (npages - 1) * kBlock < kBlock;  // the last page has rows past len
      for (int k = 0; k <= ngr; ++k) {
        if (k < ngr) {
          const int gs = k % C::NS;
          // the first group's wait may carry a shorter limit (first_wait_limit: the abort path's test)
          const uint32_t lim = (k == 0 && p.first_wait_limit != 0)
                                   ? (p.first_wait_limit < 0 ? 0u : static_cast<uint32_t>(p.first_wait_limit))
                                   : kUmmaWaitLimit;
          if (!__all_sync(0xffffffffu, umma_wait(full0 + 8 * gs, (k / C::NS) & 1, abort, lim))) break;
          if (k == 0 && p.q_tma && !__all_sync(0xffffffffu, umma_wait(qfull, 0, abort))) break;
          umma::fence_after();
          const uint64_t kd = kd0 + ((gs * C::GP * C::BOXB) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
              // 16-element k step j: box j / 4, 32 bytes per step within the 128-byte row
              umma::mma_ss(tt + 64u * (k & 1), qd + (((j >> 2) * C::QBOX + 32 * (j & 3)) >> 4),
                           kd + (((j >> 2) * C::RING + 32 * (j & 3)) >> 4), iS, j > 0 ? 1u : 0u);
            }
            umma::commit(sfull(t, k & 1));
          }
          __syncwarp();
        }
        if (k >= 1) {
          const int kp = k - 1, gsp = kp % C::NS, bp = kp & 1;
          const int npg = min(C::GP, npages - kp * C::GP);
          if (!__all_sync(0xffffffffu, umma_wait(pfull(t, bp), (kp >> 1) & 1, abort))) break;
          // the last page's V tail is zeroed by tile 0 before it hands over its P; the other
          // tiles' last P.V waits for that on v_tail, a barrier used once (a parity wait on
          // tile 0's p_full could pass a phase early if tile 0 ran several groups behind)
          if (t > 0 && kp == ngr - 1 && vtail && !__all_sync(0xffffffffu, umma_wait(vtailb, 0, abort))) break;
          umma::fence_after();
          if (elect_one()) {
            for (int i = 0; i < npg; ++i) {
              const uint32_t phi = tt + 64u * bp + 16u * i;  // P hi: 8 columns, P lo: the next 8
              const uint64_t vd = vd0 + (((gsp * C::GP + i) * C::BOXB) >> 4);
              umma::mma_ts(tt + C::OCOL, phi, vd, iPV, (kp > 0 || i > 0) ? 1u : 0u);
              umma::mma_ts(tt + C::OCOL, phi + 8u, vd, iPV, 1u);
            }
            umma::commit(odone(t));
            if (kp + C::NS < ngr) umma::commit(empty0 + 8 * gsp);  // only slots that are refilled
          }
          __syncwarp();
        }
      }
    }
  } else if (tile < ntiles) {
    // ------------------------------------------------------------ softmax (row = tid)
    const int pos = valid ? pos0 + row / G : -1;
    const float ab = (p.alibi && valid) ? __ldg(p.alibi + g * G + row % G) * 1.4426950408889634f : 0.f;
    float m = kUmmaEmpty;
    for (int k = 0; k < ngr && ok; ++k) {
      const int b = k & 1;
      if (!__all_sync(0xffffffffu, umma_wait(sfull(tile, b), (k >> 1) & 1, abort))) {
        ok = false;
        break;
      }
      umma::fence_after();
      float x[64];
      {
        float h0[32], h1[32];
        umma::ld32x2(tl + 64u * b, h0, h1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = h0[i];
          x[32 + i] = h1[i];
        }
      }
      // ---- logits in log2 units, masked past the row's position; a group the whole warp
      // sees in full (or rows without a query) skips the mask
      const int t0 = k * C::GP * kBlock;
      const bool whole = __all_sync(0xffffffffu, t0 + 63 <= pos || !valid);
      const float base = ab * static_cast<float>(t0 - pos);  // ALiBi bias of token t0
      // raw: the scores stay unscaled (scale > 0 keeps their order) and the scale is folded
      // into the exponent below; otherwise x holds the biased / masked log2 logits
      const bool raw = whole && !p.alibi;
      if (whole) {
        if (p.alibi) {
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = fmaf(x[i], p.scale_log2, fmaf(ab, static_cast<float>(i), base));
        }
      } else {
        const int lim = pos - t0;  // tokens i <= lim are visible
#pragma unroll
        for (int i = 0; i < 64; ++i)
          x[i] = i <= lim ? fmaf(x[i], p.scale_log2, fmaf(ab, static_cast<float>(i), base)) : -INFINITY;
      }
      // row max of the group: a tree of three-input max instructions
      float lm;
      {
        float a[22], b[8];
#pragma unroll
        for (int i = 0; i < 21; ++i) a[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
        a[21] = x[63];
#pragma unroll
        for (int i = 0; i < 7; ++i) b[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
        b[7] = a[21];
        lm = fmax3(fmax3(b[0], b[1], b[2]), fmax3(b[3], b[4], b[5]), fmaxf(b[6], b[7])) * (raw ? p.scale_log2 : 1.f);
      }
      const float sc = raw ? p.scale_log2 : 1.f;  // p = exp2(x sc - m)
      const bool need = lm > m + kUmmaSlack;
      const float mn = need ? lm : m;
      // P.V of the previous group must have completed before O is rescaled.  The wait is
      // unambiguous without one in every group: S(k) was issued after P.V(k - 2), so its
      // completion means at least k - 1 phases of o_done, and P.V(k) needs this group's P
      if (k >= 1 && __any_sync(0xffffffffu, need)) {
        if (!__all_sync(0xffffffffu, umma_wait(odone(tile), (k - 1) & 1, abort))) {
          ok = false;
          break;
        }
        umma::fence_after();
        const float al = ex2(m - mn);
        l *= al;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          umma::ld32(tl + C::OCOL + 32u * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= al;
          umma::st32(tl + C::OCOL + 32u * c, o);
        }
        umma::wait_st();
      }
      m = mn;
      // probabilities two at a time: exponent arguments and the row sum as packed fp32 pairs,
      // each P pair split into its 16-bit hi half and the rounded remainder (lo)
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
      const uint64_t sc2 = f2pack(sc, sc), nm2 = f2pack(-m, -m), neg1 = f2pack(-1.f, -1.f);
#pragma unroll
      for (int pg = 0; pg < C::GP; ++pg) {
        uint32_t w[16];  // 8 hi words, then 8 lo words, of the page's 16 tokens
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 e = f2unpack(f2fma(f2pack(x[16 * pg + 2 * i], x[16 * pg + 2 * i + 1]), sc2, nm2));
          const float u = ex2(e.x), v = ex2(e.y);
          const uint64_t uv = f2pack(u, v);
          ls2[i & 3] = f2add(ls2[i & 3], uv);
          float2 f;
          if constexpr (C::BF) {
            w[i] = pack_bf16(u, v);
            f = unpack_bf16(w[i]);
          } else {
            w[i] = pack_f16(u, v);
            f = unpack_f16(w[i]);
          }
          const float2 r = f2unpack(f2fma(f2pack(f.x, f.y), neg1, uv));  // (u, v) - hi, exact
          w[8 + i] = C::BF ? pack_bf16(r.x, r.y) : pack_f16(r.x, r.y);
        }
        umma::st16(tl + 64u * b + 16u * pg, w);
      }
      {
        const float2 a = f2unpack(f2add(ls2[0], ls2[1])), c = f2unpack(f2add(ls2[2], ls2[3]));
        l += (a.x + a.y) + (c.x + c.y);
      }
      umma::wait_st();
      if (k == ngr - 1 && tile == 0) {
        // V rows of tokens >= len in the last page may hold anything (NaN included) and
        // P . V would carry it into O even with P = 0 there: tile 0 zeroes them before it
        // hands over its P (the P . V of every tile is issued after that)
        const int lastp = npages - 1, nv = min(kBlock, len - lastp * kBlock);
        if (nv < kBlock) {
          const int slot = (k % C::NS) * C::GP + (lastp - k * C::GP);
          const int chunks = (kBlock - nv) * 8 * C::NBOX;  // 16-byte chunks
          for (int c = tid; c < chunks; c += 128) {
            const int bx = c / ((kBlock - nv) * 8), rr = (c / 8) % (kBlock - nv) + nv, ch = c % 8;
            *reinterpret_cast<uint4 *>(sgen + C::VOFF + bx * C::RING + slot * C::BOXB + rr * 128 + ch * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          mbar_arrive(vtailb);
        }
      }
      umma::fence_before();
      mbar_arrive(pfull(tile, b));
    }
  }
  // every role has left its loop (a block-table error it found is visible from here on)
  umma::fence_before();
  __syncthreads();
  if (*abort) {
    // A role gave up (final from here on: every role has left its loop).  Copies and MMAs may
    // still be in flight: the producer waits (bounded) for the latest group of every ring slot,
    // each MMA issuer for the completion of every MMA it issued, before the shared memory and
    // the tensor memory are released.
    if (warp == C::TMA_WARP) {
      if (lane == 0) {
        for (int k2 = max(0, issued - C::NS); k2 < issued; ++k2)
          mbar_wait_bounded(full0 + 8 * (k2 % C::NS), (k2 / C::NS) & 1, kUmmaWaitLimit);
        if (p.q_tma) mbar_wait_bounded(qfull, 0, kUmmaWaitLimit);
      }
    } else if (warp >= C::MMA_WARP && warp - C::MMA_WARP < ntiles) {
      const int t = warp - C::MMA_WARP;
      if (elect_one()) umma::commit(drain(t));  // arrives once every MMA of this issuer has completed
      __syncwarp();
      mbar_wait_bounded(drain(t), 0, kUmmaWaitLimit);
    }
  }
  if (warp < 4 * T && tile < ntiles) {
    // ---- epilogue: O / l -> out, staged in the tile's Q tile (free once the tile's last MMA
    // has completed) so that the copy to out writes whole rows with consecutive lanes
    uint8_t *stage = sgen + C::QOFF + tile * C::QTILE;
    if (ok && __all_sync(0xffffffffu, umma_wait(odone(tile), (ngr - 1) & 1, abort))) {
      umma::fence_after();
      const int rr = tid & 127;  // this thread's row within the tile
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        umma::ld32(tl + C::OCOL + 32u * c, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = C::BF ? pack_bf16(o[2 * i] * inv, o[2 * i + 1] * inv) : pack_f16(o[2 * i] * inv, o[2 * i + 1] * inv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ch = 4 * c + i;  // 16-byte chunk of the row, 128-byte swizzle as for Q
          *reinterpret_cast<uint4 *>(stage + (ch >> 3) * C::QBOX + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                     (((ch & 7) ^ (rr & 7)) << 4)) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
    // all four warps of the tile arrive here (named barrier 2 + tile); without an abort every
    // one of them staged its rows
    if (tile == 0)
      asm volatile("bar.sync 2, 128;" ::: "memory");
    else
      asm volatile("bar.sync 3, 128;" ::: "memory");
    if (!*abort && !*bad_block) {
      constexpr int CPR = D / 8;  // 16-byte chunks per row: a warp writes 512 contiguous bytes per step
      const int wl = tid & 127;
#pragma unroll 4
      for (int it = 0; it < CPR; ++it) {
        const int idx = it * 128 + wl, rr = idx / CPR, ch = idx % CPR;
        const int r = r0 + tile * 128 + rr;  // row of the KV head
        if (r - r0 < nrows) {
          const uint4 v = *reinterpret_cast<const uint4 *>(stage + (ch >> 3) * C::QBOX + (rr >> 3) * 1024 +
                                                           (rr & 7) * 128 + (((ch & 7) ^ (rr & 7)) << 4));
          OutT *dst = static_cast<OutT *>(p.out) +
                      (static_cast<int64_t>(a) + r / G) * p.out_ss + static_cast<int64_t>(g * G + r % G) * p.out_hs;
          reinterpret_cast<uint4 *>(dst)[ch] = v;
        }
      }
    }
  }
  umma::fence_before();
  __syncthreads();
  if (*abort && tid == 0 && p.err) atomicOr(p.err, kErrTimeout);
  if (warp == C::MMA_WARP) {
    umma::fence_after();
    umma::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int KIND, int D, int T>
struct UmmaLaunch {
  using C = UmmaCfg<KIND, D, T>;
  static cudaError_t launch(const DecodeParams &p, const CUtensorMap &tmK, const CUtensorMap &tmV,
                            const CUtensorMap &tmQ, cudaStream_t st) {
    auto kern = chunk_umma_kernel<KIND, D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int rows = p.nq_max * p.G;
    const dim3 grid((rows + C::ROWS - 1) / C::ROWS, p.Hkv, p.S);
    e = launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, st, 1, p, tmK, tmV, tmQ);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
};

}  // namespace pa
