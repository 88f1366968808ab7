// gdr_kkt_solve.cu - GB300 (sm_103a) fused chunk-forward kkt_solve of Gated DeltaNet.
//
// Computes, for every 64-token chunk and head, X = (I + A)^{-1} with
//   A[i][j] = beta_i * (k_i . k_j) * exp(g_i - g_j)   (j < i < L), 0 otherwise,
// and writes X as out[B, T, H, 64] (MindSpeed-Ops PR #135 page, "feat(triton): add
// chunk_gated_delta_rule_fwd_kkt_solve", section "What this PR does": one call
// replaces solve_tril(chunk_scaled_dot_kkt_fwd(...)); API block: result
// (I+A)^{-1} of shape [B, T, H, 64]).  The intermediate A never leaves the SM
// and no separate zero-fill pass runs.
//
// Kernel organisation (one persistent CTA per SM, 14 warps; a CTA takes the tile
// pairs blockIdx.x, blockIdx.x + grid, ...):
//   warp 12      producer: lanes 0-1 TMA-load the key tiles of the next pair's two
//                (chunk, head) tiles into a three-stage ring (bf16, 128-byte
//                swizzle, 32 KB per stage); lanes 2-3 prefetch into L2 the keys of
//                the pair two steps further on.
//   warp 13      MMA issuer: allocates TMEM and, per stage, issues tcgen05.mma
//                (kind::f16, M = N = 128 = both tiles' rows, K = 128 in 8 steps),
//                so TMEM holds the pair's 128 x 128 Gram matrix in fp32; each tile
//                reads its own 64 x 64 diagonal block.
//   warps 0..11  three consumer warpgroups; each owns 128 TMEM columns and one
//                tile pair at a time:
//                  epilogue - each thread reads its row of S = K*K^T from TMEM,
//                             applies beta_i and exp(g_i - g_j) (exponent clamped
//                             to [-50, 50] as in the page's bot summary) and writes
//                             row i of A to shared memory (fp32);
//                  solve    - the page's 16 x 16 sub-blocks (BC = 16): the four
//                             diagonal inverses by substitution on CUDA cores (one
//                             lane per row), the six blocks below them on tensor
//                             cores (mma.sync tf32);
//                  store    - X is assembled in a 128-byte-swizzled staging copy
//                             and written by TMA (full chunks) or by 128-bit
//                             stores (a chunk cut short by the sequence end).
// The same template also builds: fp16 keys and K = 64..256 (the key type only
// changes the TMA map and the MMA descriptor; K / 64 sets the stage units per
// pair); fp32 keys (bf16 output: one tf32 product on the keys as loaded;
// fp32 or fp16 output: two more warps split each unit into tf32 parts for a
// three-product tf32 Gram); the two halves of the page's unfused chain (A
// written to HBM; the solve of a given A).  kkt_solve_c128_kernel handles
// 128-token chunks.
// Every mbarrier wait is bounded by wall time; on expiry the kernel records
// GDR_ERR_TIMEOUT in a device status word and all roles leave their loops.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <stdint.h>

#include "gdr_kkt_solve.h"

namespace gdr {

constexpr int kChunk = 64;
constexpr int kMaxHeadK = 256;                    // K = 64, 128, 192 or 256

constexpr int kBoxBytes = kChunk * 64 * 2;          // one (tile, K-half) box: 64 rows x 128 B
constexpr int kStageBytes = 4 * kBoxBytes;          // [K-half][tile][64 rows][128 B] = 32 KB
// Row r of a 64 x 64 fp32 matrix (A, then X) in shared memory starts at float
// a_row<P>(r): P = 72 puts it at 72 r + (r & 4), P = 68 at 68 r (see a_row).
// The 64-token kernel takes P = 72 for bf16 output and 68 otherwise (there the
// wider rows cost registers the split merge needs); its buffers fit either.
constexpr int kAPitch = 72;                         // the larger row pitch, for buffer sizes
constexpr int kATileBytes = kChunk * kAPitch * 4;   // 18432
constexpr int kATile1Off = kATileBytes;
constexpr int kAWGBytes = 36864;                    // >= kATile1Off + kATileBytes, multiple of 1024
constexpr int kStage1Off = 17408;                   // output staging of the second tile (1024-aligned)
constexpr int kGWGBytes = 2 * 2 * 2 * kChunk * 4;   // g and v of two tiles, double buffered
constexpr uint32_t kTmemCols = 512;
// L2 prefetch distance of the key tiles, in pairs: the producer's lanes 2 and
// 3 issue cp.async.bulk.prefetch for pair q + d while lanes 0 and 1 load pair
// q.  With d = 0 the prefetch goes out as soon as the producer reaches a pair,
// ahead of its wait for a free stage; measured over d = -1 (none) .. 4 on
// (2, 16384, 32, K), d = 0 is fastest where a pair's keys are one stage unit
// (and for the chunk-128 kernel and the split fp32-key Gram) and d = 1 where
// they are two 128-column units (K = 192, 256; fp32 keys as loaded, K = 128).
__host__ __device__ constexpr int prefetch_pairs(int units_per_pair, bool split_f32) {
    return units_per_pair == 2 && !split_f32 ? 1 : 0;
}

constexpr int kOffK = 0;

constexpr uint64_t kWaitNs = 2000000000ull;         // 2 s bound for every wait
constexpr uint32_t kSuspendNs = 1000000;             // a waiting thread sleeps until the phase completes (or 1 ms)

// Division by an invariant divisor d >= 1 for numerators n < 2^31 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994): with
// l = ceil(log2 d) and m = ceil(2^(31+l) / d), floor(n / d) = (n * m) >> (31 + l);
// m < 2^33, so the product fits in 64 bits.
struct FastDiv {
    uint64_t m;
    uint32_t shift;
    uint32_t d;
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return static_cast<uint32_t>((static_cast<uint64_t>(n) * m) >> shift);
    }
};

inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    FastDiv f;
    f.d = d;
    f.shift = 31 + l;
    f.m = ((uint64_t(1) << f.shift) + d - 1) / d;
    return f;
}

struct Params {
    const float *g;
    const void *beta;
    const int32_t *cu;
    void *out;
    int64_t B, T, H;
    int64_t n_slots;   // chunk slots: fixed-length B*NT, varlen floor((T + 63 B)/64)
    int64_t NT;        // chunks per sequence (fixed-length)
    int64_t n_pairs;   // ceil(n_slots * H / 2)
    FastDiv divH;      // tile -> (slot, head)
    FastDiv divNT;     // slot -> (sequence, chunk), fixed-length
    uint32_t pair_ds, pair_dh;   // stride between a CTA's consecutive pairs (2 * grid tiles) as (slots, heads)
    uint32_t wg_ds, wg_dh;       // stride between a warpgroup's consecutive pairs (2 * grid * warpgroups tiles)
    int *status;
    uint32_t idesc;    // tcgen05 instruction descriptor for the key type
    int beta_kind;     // gdr_dtype of beta (GDR_F32 when beta is NULL)
};

struct Tile {
    int64_t row0;      // first token row of the chunk in the flattened token axis
    int L;             // rows in the chunk; 0 = no tile
    int h;
};

__device__ int g_status_word = 0;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete; false after LIMIT ns.
template <uint64_t LIMIT>
__device__ __noinline__ bool mbar_wait_limited(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer() - t0 > LIMIT) return false;
    }
}
// The first (suspend-hinted) try_wait is inline, the bounded retry loop out of
// line: most waits end in the first try_wait, and a call per wait measured
// 1.9 % on (2, 16384, 32, 128) bf16.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_limited<kWaitNs>(bar, parity);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// Programmatic dependent launch: the grid may start while the previous grid on
// the stream is still finishing (it is launched with programmatic stream
// serialization).  Nothing may touch global memory before grid_dependency_wait
// returns, which happens once every prerequisite grid has completed and its
// writes are visible; grid_launch_dependents lets the next grid's CTAs begin
// their own set-up as this grid's CTAs exit.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Ties registers written by tcgen05.ld to a point after tcgen05.wait::ld, so the
// compiler cannot hoist their first use above the wait.
__device__ __forceinline__ void reg_fence(uint32_t &r) { asm volatile("" : "+r"(r)); }

// Shared-memory matrix descriptor of a K-major bf16 operand stored as 8-row x
// 128-byte swizzle atoms (the layout a 128-byte-swizzled TMA box produces):
// start address, leading offset (unused for this layout), stride between 8-row
// groups = 1024 B, descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B of the key type (format 1 =
// bf16, 0 = fp16), both K-major, N = 128, M = 128.
// kind::tf32: D fp32, A and B tf32 (format 2), both K-major, N = 128, M = 128.
constexpr uint32_t kIdescTf32 = (1u << 4) | (2u << 7) | (2u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t idesc_f16_kind(bool bf16_keys) {
    return (1u << 4) | ((bf16_keys ? 1u : 0u) << 7) | ((bf16_keys ? 1u : 0u) << 10) |
           ((128u >> 3) << 17) | ((128u >> 4) << 24);
}
constexpr uint32_t kIdescBf16 = idesc_f16_kind(true);

// ------------------------------------------------------------ tile schedule
// Tile u = slot * H + h.  Fixed-length: slot = b * NT + c.  Varlen: sequence n
// owns the slots [base(n), base(n+1)) with base(n) = floor((cu[n] + 63 n) / 64),
// which leaves room for its ceil(len/64) chunks (at most one slot stays empty).
// The tiles a role visits form an arithmetic sequence u, u + S, u + 2S, ...
// (S = 2 * grid tiles for the producer's pairs, 2 * grid * warpgroups for one
// warpgroup's).  TileWalk keeps u's (slot, h) and the slot's (sequence, chunk)
// and steps them by S = ds * H + dh with one carry: fixed-length moves the chunk
// index and divides only when it passes NT; varlen moves the sequence index
// forward over the boundaries base(n + 1) the slot has passed (base is
// non-decreasing in n, so this finds the same sequence as a binary search).
struct TileWalk {
    uint32_t slot, h;
    uint32_t b, c;          // fixed-length: slot = b * NT + c
    int32_t n, s, e;        // varlen: sequence n of the slot, cu[n], cu[n + 1]
    int64_t bn1;            // varlen: base(n + 1)
};

// CH is the chunk length (64, or 128 for the chunk-128 kernel, whose "tiles" are
// whole chunks).
template <int CH>
constexpr int kLog2 = CH == 64 ? 6 : 7;

template <int CH = kChunk>
__device__ __forceinline__ TileWalk walk_init(const Params &p, uint32_t u) {
    TileWalk w;
    w.slot = p.divH.div(u);
    w.h = u - w.slot * p.divH.d;
    w.b = w.c = 0;
    w.n = static_cast<int32_t>(p.B);
    w.s = w.e = 0;
    w.bn1 = 0;
    if (p.cu == nullptr) {
        w.b = p.divNT.div(w.slot);
        w.c = w.slot - w.b * p.divNT.d;
    } else if (w.slot < static_cast<uint64_t>(p.n_slots)) {
        int64_t lo = 0, hi = p.B;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            const int64_t bm = (static_cast<int64_t>(__ldg(p.cu + mid)) + (CH - 1) * mid) >> kLog2<CH>;
            if (bm <= w.slot) lo = mid;
            else hi = mid - 1;
        }
        w.n = static_cast<int32_t>(lo);
        if (lo < p.B) {
            w.s = __ldg(p.cu + lo);
            w.e = __ldg(p.cu + lo + 1);
            w.bn1 = (static_cast<int64_t>(w.e) + (CH - 1) * (lo + 1)) >> kLog2<CH>;
        }
    }
    return w;
}

template <int CH = kChunk>
__device__ __forceinline__ void walk_advance(const Params &p, TileWalk &w, uint32_t ds, uint32_t dh) {
    uint32_t inc = ds;
    w.h += dh;
    if (w.h >= p.divH.d) {
        w.h -= p.divH.d;
        ++inc;
    }
    w.slot += inc;
    if (p.cu == nullptr) {
        w.c += inc;
        if (w.c >= p.divNT.d) {
            const uint32_t qd = p.divNT.div(w.c);
            w.b += qd;
            w.c -= qd * p.divNT.d;
        }
    } else {
        // At most B steps over the whole walk; never reads past cu[B].
        while (w.n < p.B && w.bn1 <= static_cast<int64_t>(w.slot)) {
            ++w.n;
            w.s = w.e;
            if (w.n < p.B) {
                w.e = __ldg(p.cu + w.n + 1);
                w.bn1 = (static_cast<int64_t>(w.e) + (CH - 1) * static_cast<int64_t>(w.n + 1)) >> kLog2<CH>;
            }
        }
    }
}

template <int CH = kChunk>
__device__ __forceinline__ Tile walk_tile(const Params &p, const TileWalk &w) {
    Tile t;
    t.row0 = 0;
    t.L = 0;
    t.h = static_cast<int>(w.h);
    if (w.slot >= static_cast<uint64_t>(p.n_slots)) return t;
    if (p.cu == nullptr) {
        t.row0 = static_cast<int64_t>(w.b) * p.T + static_cast<int64_t>(w.c) * CH;
        const int64_t rem = p.T - static_cast<int64_t>(w.c) * CH;
        t.L = static_cast<int>(rem < CH ? rem : CH);
        return t;
    }
    if (w.n >= p.B) return t;
    const int64_t s = w.s;
    const int64_t e = w.e > p.T ? p.T : w.e;
    const int64_t c = static_cast<int64_t>(w.slot) - ((s + (CH - 1) * static_cast<int64_t>(w.n)) >> kLog2<CH>);
    const int64_t r0 = s + c * CH;
    if (c < 0 || s < 0 || r0 >= e) return t;
    t.row0 = r0;
    t.L = static_cast<int>(e - r0 < CH ? e - r0 : CH);
    return t;
}

// ------------------------------------------------------------- the inverse
// X = (I + A)^{-1} is built from 16x16 blocks (the page's BC = 16 sub-blocks):
//   D_II = (I + A_II)^{-1}                       for the four diagonal blocks,
//   X_IJ = -D_II * sum_{M=J}^{I-1} A_IM X_MJ     for the six blocks below them.
// The diagonal blocks use fp32 forward substitution on CUDA cores (one lane per
// row).  The off-diagonal products run on tensor cores with mma.sync tf32: for
// fp32 output as 3xTF32 (x = big + small, both tf32; big*big + big*small +
// small*big), which keeps them fp32-accurate; for bf16 output as one tf32
// pass, whose error (max ~2e-4 on the workloads, fp64 emulation) is below the
// bf16 rounding of the result.  They are evaluated transposed, Z_JI = X_IJ^T =
// -(sum_M Z_JM A_IM^T) D_II^T, so every product's left operand is the previous
// product's accumulator.

// Bank layout of the matrix rows.  With P = 72 rows start 72 r + (r & 4) floats
// apart: eight consecutive rows begin in eight different 4-bank groups (the
// row-per-lane float4 writes and reads), and the merge's float2 operand reads
// (rows 8 nt + g of one half-warp, columns 2 t, 2 t + 1) cover all 32 banks; its
// transposed scalar reads (rows 2 t and 2 t + 1, columns g) are 2-way.  With
// P = 68 the scalar reads are conflict-free and the float2 reads 2-way; the
// chunk-128 kernel (no room for wider rows) and the 64-token kernel's fp32 and
// fp16 outputs (whose split merge needs the registers the wider addressing
// takes) keep it.  A block row r0 + x with r0 a multiple of 16 starts at
// a_row(r0) + a_row(x) in both layouts.
template <int P>
__device__ __forceinline__ int a_row(int r) {
    static_assert(P == 68 || P == 72, "matrix row layouts");
    return P == 72 ? r * 72 + (r & 4) : r * 68;
}

// Diagonal inverses are parked in the free upper blocks of the A buffer:
// D_00 -> block (0,1), D_11 -> (0,2), D_22 -> (0,3), D_33 -> (1,2).
__device__ __forceinline__ int dslot_r(int I) { return I == 3 ? 1 : 0; }
__device__ __forceinline__ int dslot_c(int I) { return I == 3 ? 2 : I + 1; }

// Row c of D_II by right-looking substitution inside block (I, I): y[j]
// accumulates -sum_{i>j} A[i][j] y[i]; processing i downwards, y[i] is final
// (plus 1 on the diagonal) when reached.  Rows above c give y = 0.
template <int P>
__device__ __forceinline__ void diag_inverse_row(const float *Ab, int c, float (&y)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) y[j] = 0.0f;
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
        const int i = 15 - ii;
        y[i] += (i == c) ? 1.0f : 0.0f;
        const float yi = y[i];
        const float4 *Ar = reinterpret_cast<const float4 *>(Ab + a_row<P>(i));
#pragma unroll
        for (int j4 = 0; j4 < (i + 3) / 4; ++j4) {
            const float4 a = Ar[j4];
            if (4 * j4 + 0 < i) y[4 * j4 + 0] = fmaf(-a.x, yi, y[4 * j4 + 0]);
            if (4 * j4 + 1 < i) y[4 * j4 + 1] = fmaf(-a.y, yi, y[4 * j4 + 1]);
            if (4 * j4 + 2 < i) y[4 * j4 + 2] = fmaf(-a.z, yi, y[4 * j4 + 2]);
            if (4 * j4 + 3 < i) y[4 * j4 + 3] = fmaf(-a.w, yi, y[4 * j4 + 3]);
        }
    }
}

// A 16x16 fp32 left operand in m16n8k8 A-fragment layout for both k8 steps,
// split into tf32 big and small parts.  Inside each k8 step the k order is
// permuted (logical k = t -> column 2t, k = t + 4 -> column 2t + 1); with that
// order an m16n8 accumulator pair is already a left operand.  Every right
// operand below uses the same order.
struct Frag16 {
    uint32_t big[2][4];
    uint32_t small[2][4];
};

// x = big + small exactly: big is x rounded to tf32 (ten mantissa bits, round
// half away from zero, done on the bit pattern: add half an ulp of tf32, clear
// the 13 low bits), small = x - big with |small| <= 2^-11 |x|; the tensor core
// reads small to tf32 precision, so the split products carry ~2^-21 relative
// error.  Integer arithmetic keeps the split on the full-rate ALU pipes.
__device__ __forceinline__ void split_tf32(float x, uint32_t &big, uint32_t &small) {
    const uint32_t b = (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
    big = b;
    small = __float_as_uint(x - __uint_as_float(b));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// SPLIT = false keeps the raw fp32 bits in f.big (the tensor core reads them as
// tf32) for a single-pass product; f.small is unused then.
template <bool SPLIT>
__device__ __forceinline__ void frag_from_acc(const float (&acc)[2][4], Frag16 &f) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const float v[4] = {acc[ks][0], acc[ks][2], acc[ks][1], acc[ks][3]};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (SPLIT) split_tf32(v[e], f.big[ks][e], f.small[ks][e]);
            else f.big[ks][e] = __float_as_uint(v[e]);
        }
    }
}

// acc += F * Bm for a 16x16 right operand Bm read from shared memory: for k8
// step ks, n8 tile nt and this lane (g = lane / 4, t = lane % 4) the pair
// (Bm[8ks + 2t][8nt + g], Bm[8ks + 2t + 1][8nt + g]) is the float2 in block row
// 8 nt + g at column 8 ks + 2 t, i.e. Bm is the transpose of the row-major
// 16x16 block at rowp.
template <bool SPLIT, int P>
__device__ __forceinline__ void mma3_times_blockT(float (&acc)[2][4], const Frag16 &f,
                                                  const float *rowp, int g, int t) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float2 b = *reinterpret_cast<const float2 *>(rowp + a_row<P>(8 * nt + g) + 8 * ks + 2 * t);
            if (SPLIT) {
                uint32_t bb0, bs0, bb1, bs1;
                split_tf32(b.x, bb0, bs0);
                split_tf32(b.y, bb1, bs1);
                mma_tf32(acc[nt], f.small[ks], bb0, bb1);
                mma_tf32(acc[nt], f.big[ks], bs0, bs1);
                mma_tf32(acc[nt], f.big[ks], bb0, bb1);
            } else {
                mma_tf32(acc[nt], f.big[ks], __float_as_uint(b.x), __float_as_uint(b.y));
            }
        }
    }
}

// Left operand D_JJ^T (= Z_JJ) read from its parking block.
template <bool SPLIT, int P>
__device__ __forceinline__ void frag_from_dT(const float *D, int g, int t, Frag16 &f) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        // Row 8 ks + 2 t is even, so the next row starts P floats later in both layouts.
        float v[4];
        if constexpr (P == 68) {
            v[0] = D[(8 * ks + 2 * t) * P + g];
            v[1] = D[(8 * ks + 2 * t) * P + g + 8];
            v[2] = D[(8 * ks + 2 * t + 1) * P + g];
            v[3] = D[(8 * ks + 2 * t + 1) * P + g + 8];
        } else {
            const float *r0 = D + a_row<P>(8 * ks + 2 * t);
            v[0] = r0[g];
            v[1] = r0[g + 8];
            v[2] = r0[P + g];
            v[3] = r0[P + g + 8];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (SPLIT) split_tf32(v[e], f.big[ks][e], f.small[ks][e]);
            else f.big[ks][e] = __float_as_uint(v[e]);
        }
    }
}

// Blocks Z_JI = X_IJ^T for I = J+1..3 of one tile (At = its A buffer).  Split
// operands are rebuilt when needed instead of cached, to stay within registers.
template <int J, bool SPLIT, int P>
__device__ __forceinline__ void merge_column(const float *At, int g, int t,
                                             float (&Z)[3 - J][2][4]) {
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
        float acc[2][4] = {};
#pragma unroll
        for (int M = J; M < I; ++M) {
            Frag16 f;
            if (M == J) frag_from_dT<SPLIT, P>(At + a_row<P>(16 * dslot_r(J)) + 16 * dslot_c(J), g, t, f);
            else frag_from_acc<SPLIT>(Z[M - J - 1], f);
            mma3_times_blockT<SPLIT, P>(acc, f, At + a_row<P>(16 * I) + 16 * M, g, t);
        }
        Frag16 rf;
        frag_from_acc<SPLIT>(acc, rf);
        float z[2][4] = {};
        mma3_times_blockT<SPLIT, P>(z, rf, At + a_row<P>(16 * dslot_r(I)) + 16 * dslot_c(I), g, t);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) Z[I - J - 1][nt][e] = -z[nt][e];
    }
}

// ------------------------------------------------------------ output staging
// X is assembled in the layout a 128-byte-swizzled TMA store reads: a tile's 64
// rows of 128 bytes (bf16: 64 values; fp32: two 32-value halves 8 KB apart), the
// 16-byte piece q of row r stored at piece position q ^ (r % 8).
template <bool OUT16>
__device__ __forceinline__ uint32_t stage_piece_off(int r, int q) {
    if (OUT16) return static_cast<uint32_t>(r * 128 + ((q ^ (r & 7)) << 4));
    return static_cast<uint32_t>((q >> 3) * 8192 + r * 128 + (((q & 7) ^ (r & 7)) << 4));
}

// One fp32 value of X at (r, c) in the fp32 staging.
__device__ __forceinline__ void stage_put_f32(uint8_t *st, int r, int c, float v) {
    *reinterpret_cast<float *>(st + stage_piece_off<false>(r, c >> 2) + 4 * (c & 3)) = v;
}

// Output kinds (the gdr_dtype values): fp32, bf16, fp16.  The 16-bit kinds share
// the staging layout and differ only in the rounding to 16 bits (both
// round-to-nearest-even); a holds the lower column.
constexpr int kOutF32 = 0, kOutBF16 = 1, kOutF16 = 2;
template <int OUT>
__device__ __forceinline__ uint32_t pack16x2(float a, float b) {
    if (OUT == kOutF16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Row r of X restricted to columns >= 16 I: the diagonal block row (d[0..3] =
// 16 values) followed by zeros.
template <int OUT>
__device__ __forceinline__ void stage_diag_row(uint8_t *st, int r, int I, const float4 (&d)[4]) {
    if (OUT != kOutF32) {
        uint4 a, b;
        a.x = pack16x2<OUT>(d[0].x, d[0].y); a.y = pack16x2<OUT>(d[0].z, d[0].w);
        a.z = pack16x2<OUT>(d[1].x, d[1].y); a.w = pack16x2<OUT>(d[1].z, d[1].w);
        b.x = pack16x2<OUT>(d[2].x, d[2].y); b.y = pack16x2<OUT>(d[2].z, d[2].w);
        b.z = pack16x2<OUT>(d[3].x, d[3].y); b.w = pack16x2<OUT>(d[3].z, d[3].w);
        *reinterpret_cast<uint4 *>(st + stage_piece_off<true>(r, 2 * I)) = a;
        *reinterpret_cast<uint4 *>(st + stage_piece_off<true>(r, 2 * I + 1)) = b;
#pragma unroll
        for (int q = 2; q < 8; ++q)
            if (q >= 2 * I + 2) *reinterpret_cast<uint4 *>(st + stage_piece_off<true>(r, q)) = make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
        for (int m = 0; m < 4; ++m)
            *reinterpret_cast<float4 *>(st + stage_piece_off<false>(r, 4 * I + m)) = d[m];
#pragma unroll
        for (int q = 4; q < 16; ++q)
            if (q >= 4 * I + 4)
                *reinterpret_cast<float4 *>(st + stage_piece_off<false>(r, q)) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Z_JI (accumulator layout) -> rows 16I.. / columns 16J.. of X in the staging.
// 16-bit output: one transposing matrix store; the accumulator pairs (z[nt][0], z[nt][1])
// and (z[nt][2], z[nt][3]) are the fragments of four 8x8 matrices, stored
// transposed, whose rows (X rows 16I + 8 (m / 2) + b, 16-byte piece 2J + m % 2)
// are addressed by lane 8m + b.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1,
                                                  uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}
template <int OUT>
__device__ __forceinline__ void stage_block_T(uint8_t *st, int I, int J, const float (&z)[2][4],
                                              int g, int t) {
    if (OUT != kOutF32) {
        const int lane = 4 * g + t, m = lane >> 3, b = lane & 7;
        const uint32_t addr = smem_u32(st + stage_piece_off<true>(16 * I + 8 * (m >> 1) + b, 2 * J + (m & 1)));
        stmatrix_x4_trans(addr, pack16x2<OUT>(z[0][0], z[0][1]), pack16x2<OUT>(z[0][2], z[0][3]),
                          pack16x2<OUT>(z[1][0], z[1][1]), pack16x2<OUT>(z[1][2], z[1][3]));
    } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int r0 = 16 * I + 8 * nt + 2 * t, c0 = 16 * J + g;
            stage_put_f32(st, r0, c0, z[nt][0]);
            stage_put_f32(st, r0 + 1, c0, z[nt][1]);
            stage_put_f32(st, r0, c0 + 8, z[nt][2]);
            stage_put_f32(st, r0 + 1, c0 + 8, z[nt][3]);
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Writes Z_JI (accumulator layout) into rows 16I.. / columns 16J.. of X.
template <int P>
__device__ __forceinline__ void store_block_T(float *At, int I, int J, const float (&z)[2][4],
                                              int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        float *r0 = At + a_row<P>(16 * I + 8 * nt + 2 * t) + 16 * J + g;   // even row: next at + P
        r0[0] = z[nt][0];
        r0[P] = z[nt][1];
        r0[8] = z[nt][2];
        r0[P + 8] = z[nt][3];
    }
}

__device__ __forceinline__ void record_timeout(const Params &p, volatile int *abort_flag) {
    *abort_flag = 1;
    atomicExch(p.status, static_cast<int>(GDR_ERR_TIMEOUT));
}

// Per-row gate inputs of a tile, loaded one pair ahead and kept raw (no
// arithmetic on them until they are used, so the loads stay in flight): this
// row's g and beta, and the chunk's first and last g.
struct RowIn {
    float g, gfirst, glast;
    uint32_t beta;     // raw bits of beta in its own type
};

__device__ __forceinline__ RowIn load_row(const Params &p, const Tile &t, int i) {
    RowIn r;
    r.g = 0.0f;
    r.gfirst = 0.0f;
    r.glast = 0.0f;
    r.beta = 0x3F800000u;   // fp32 1.0 (beta NULL is read as fp32)
    if (i < t.L) {
        const int64_t base = t.row0 * p.H + t.h;
        if (p.g) {
            r.g = __ldg(p.g + base + static_cast<int64_t>(i) * p.H);
            r.gfirst = __ldg(p.g + base);
            r.glast = __ldg(p.g + base + static_cast<int64_t>(t.L - 1) * p.H);
        }
        if (p.beta) {
            const int64_t at = base + static_cast<int64_t>(i) * p.H;
            r.beta = p.beta_kind == GDR_F32
                         ? __ldg(reinterpret_cast<const uint32_t *>(p.beta) + at)
                         : static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p.beta) + at));
        }
    }
    return r;
}

__device__ __forceinline__ float beta_value(const Params &p, uint32_t bits) {
    if (p.beta_kind == GDR_BF16) return __uint_as_float(bits << 16);
    if (p.beta_kind == GDR_F16) return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    return __uint_as_float(bits);
}

__device__ __forceinline__ bool named_bar_red_or(int id, int nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// Modes: the fused step; its first half alone (A = beta K K^T exp(gate), strictly
// lower, written to HBM as fp32 like the page's chunk_scaled_dot_kkt_fwd); its
// second half alone ((I + A)^{-1} from that A, like the page's solve_tril).  The
// halves run the fused step's own code, so the two-kernel chain reproduces the
// fused result bit for bit.
constexpr int kModeFused = 0, kModeKkt = 1, kModeSolve = 2;
// The fused step with fp32 keys: the stage unit is one 32-column fp32 box per
// tile (NKB = K / 32 units per pair); converter warps split each key x into
// big = x rounded to tf32 and small = x - big (|small| <= 2^-11 |x|), and the
// Gram is big big^T on the kind::tf32 tensor cores plus the cross products
// bf16(big) bf16(small)^T + bf16(small) bf16(big)^T on the kind::f16 path.
// Per product x_i x_j the bf16 roundings cost at most 2 * 2^-8 * 2^-11 and the
// dropped small small^T at most 2^-22 of |x_i x_j|: about 2^-18 in all.
constexpr int kModeF32Keys = 3;
// The fused step with fp32 keys and bf16 output: the key units are the boxes of
// fp32 columns as loaded, the MMA warp issues one kind::tf32 product per K step
// on them, and no split is made.  Narrowing an fp32 key to tf32 changes it by
// at most 2^-10 of its value (truncated or rounded), which leaves the result
// within a fraction of one bf16 rounding of the output.
constexpr int kModeF32KeysTf32 = 4;

// Shared-memory plan and warp roles of the 64-token kernel, per mode.  Warps
// 0 .. 4 NWG - 1 are the consumer warpgroups, then the producer warp, the MMA
// warp and, for the split fp32-key Gram, the converter warps.  The split Gram
// needs each unit's bf16 pair operand beside its keys, and its speed is set by
// the key bytes in flight and by its converters (its consumers keep up with
// two warpgroups), so it trades the third warpgroup's buffers and registers
// for a six-unit ring of 16 KB key units, a three-unit ring of 16 KB pair
// units and four converter warps; every other mode runs three consumer
// warpgroups on a three-unit ring of 32 KB key units.
template <int MODE>
struct FusedLayout {
    static constexpr bool kSplit = MODE == kModeF32Keys;
    static constexpr int kNumWG = kSplit ? 2 : 3;
    static constexpr int kNumStages = kSplit ? 6 : 3;                 // key units
    static constexpr int kUnitBytes = kSplit ? 2 * kBoxBytes : kStageBytes;
    static constexpr int kNumRem = kSplit ? 3 : 0;                    // bf16 pair units
    static constexpr int kRemBytes = 2 * kBoxBytes;
    static constexpr int kConsumerWarps = 4 * kNumWG;
    static constexpr int kProducerWarp = kConsumerWarps;
    static constexpr int kMmaWarp = kConsumerWarps + 1;
    static constexpr int kCvtWarp0 = kConsumerWarps + 2;
    // Converter warps: kCvtGroups groups of kCvtPerGroup warps; group g splits
    // the key units v = g, g + kCvtGroups, ....  One group of four measured
    // fastest: a converter warp shares its scheduler's issue slots with
    // consumer warps, so a unit converts soonest spread over the most warps
    // (two or three groups converting whole units in turn were much slower).
    static constexpr int kCvtGroups = 1;
    static constexpr int kCvtPerGroup = 4;
    static constexpr int kCvtWarps = kSplit ? kCvtGroups * kCvtPerGroup : 0;
    static constexpr int kThreads = 32 * (kConsumerWarps + 2 + kCvtWarps);
    static constexpr int kOffRem = kOffK + kNumStages * kUnitBytes;
    static constexpr int kOffA = kOffRem + kNumRem * kRemBytes;
    static constexpr int kOffG = kOffA + kNumWG * kAWGBytes;
    static constexpr int kOffBar = kOffG + kNumWG * kGWGBytes;
    // full, empty [stages]; tfull, tempty [warpgroups]; converted, pair unit free [pair units]
    static constexpr int kNumBars = 2 * kNumStages + 2 * kNumWG + 2 * kNumRem;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 1024;           // slack for 1024-byte alignment
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffA % 1024 == 0 && kOffRem % 1024 == 0, "key units keep 1024-byte alignment");
    static_assert(kThreads <= 512, "launch shape");
};

// OUT: kOutF32, kOutBF16 or kOutF16.  The merge runs split (fp32-accurate) for
// fp32 and fp16 output and as one tf32 pass for bf16 output.  NKB = K / 64, the
// 64-column key boxes per row; it only shapes the producer and MMA loops, which
// sit on the pipeline's critical path and so are fully unrolled per K.  In the
// solve mode the producer loads A tiles (two 32-column fp32 boxes per tile,
// NKB = 2) and the MMA warp has nothing to do.
template <int OUT, int NKB, int MODE>
__global__ void __launch_bounds__(FusedLayout<MODE>::kThreads, 1)
    kkt_solve_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_out, const Params p) {
    static_assert(MODE != kModeKkt || OUT == kOutF32, "A is written as fp32");
    static_assert(MODE != kModeSolve || NKB == 2, "an A tile row is two 128-byte boxes");
    using L = FusedLayout<MODE>;
    constexpr int kNumWG = L::kNumWG;
    constexpr int kNumStages = L::kNumStages;
    constexpr int kNumRem = L::kNumRem;
    constexpr int kRemMod = kNumRem > 0 ? kNumRem : 1;   // pair-unit ring modulus (unused without a split)
    constexpr int kUnitBytes = L::kUnitBytes;
    constexpr int kProducerWarp = L::kProducerWarp;
    constexpr int kMmaWarp = L::kMmaWarp;
    constexpr int kCvtWarp0 = L::kCvtWarp0;
    constexpr bool kUseTmem = MODE != kModeSolve;
    constexpr bool kF32Keys = MODE == kModeF32Keys;
    constexpr int kP = OUT == kOutBF16 ? 72 : 68;    // A buffer row layout (a_row)
    // Elements per 128-byte box row: 64 bf16/fp16 key columns, or 32 fp32 ones.
    constexpr bool kTf32Gram = MODE == kModeF32KeysTf32;
    constexpr int kBoxCols = (MODE == kModeSolve || kF32Keys || kTf32Gram) ? 32 : 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + L::kOffBar;                    // [kNumStages]
    const uint32_t bar_empty = bar_full + 8 * kNumStages;            // [kNumStages]
    const uint32_t bar_tfull = bar_empty + 8 * kNumStages;           // [kNumWG]
    const uint32_t bar_tempty = bar_tfull + 8 * kNumWG;              // [kNumWG]
    const uint32_t bar_cvt = bar_tempty + 8 * kNumWG;                // [kNumRem], split fp32 keys
    const uint32_t bar_rfree = bar_cvt + 8 * kNumRem;                // [kNumRem], split fp32 keys
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
    volatile int *wg_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);   // [kNumWG]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNumStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            // Freed by the MMA commit, or in the solve mode by the 4 warps of the
            // warpgroup that copied the stage.
            mbar_init(bar_empty + 8 * s, kUseTmem ? 1 : 4);
        }
        for (int w = 0; w < kNumWG; ++w) {
            mbar_init(bar_tfull + 8 * w, 1);
            mbar_init(bar_tempty + 8 * w, 4);
        }
        for (int u = 0; u < kNumRem; ++u) {
            mbar_init(bar_cvt + 8 * u, L::kCvtPerGroup);
            mbar_init(bar_rfree + 8 * u, 1);     // the MMA commit
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (kUseTmem && warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = kUseTmem ? *tmem_slot : 0u;
    // Set-up above touched only shared memory and TMEM: from here on global
    // memory is read and written.
    grid_dependency_wait();
    grid_launch_dependents();

    const int64_t n_local = (p.n_pairs > blockIdx.x)
                                ? (p.n_pairs - 1 - blockIdx.x) / gridDim.x + 1
                                : 0;

    // The pipeline unit is (pair, 128-column chunk of K): K = 64 or 128 takes one
    // unit per pair, K = 192 or 256 two.  A unit holds one or two 64-column boxes
    // of each of the pair's tiles; the Gram accumulates over a pair's units.
    constexpr int nkb = NKB;
    constexpr int nkc = kF32Keys ? nkb : (nkb + 1) >> 1;
    constexpr int kPrefetchPairs = prefetch_pairs(nkc, kF32Keys);
    if (warp == kProducerWarp) {
        // Lanes 0 and 1 walk the two tiles of pair q (loaded into the stage ring),
        // lanes 2 and 3 those of pair q + kPrefetchPairs (prefetched into L2).
        // Each lane issues the copies of its own tile, so one warp instruction
        // covers all four; lane 0 owns the stage barriers.
        if (lane < 4) {
            if (lane == 0)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k))
                             : "memory");
            const int tt = lane & 1;
            const bool pf_lane = lane >= 2;
            TileWalk w = walk_init(p, static_cast<uint32_t>(2 * blockIdx.x + tt));
            if (pf_lane)
                for (int i = 0; i < kPrefetchPairs; ++i) walk_advance(p, w, p.pair_ds, p.pair_dh);
            int64_t q = 0;
            int kc = 0;             // units of pair q issued when the loop stops inside it
            bool failed = false;
            for (; q < n_local; ++q) {
                int stop = (lane == 0) ? *abort_flag : 0;
                if (__shfl_sync(0xFu, stop, 0)) break;
                const Tile t = walk_tile(p, w);
                if (pf_lane) {
                    if (q + kPrefetchPairs < n_local) {
                        if (t.L > 0)
#pragma unroll
                            for (int kb = 0; kb < nkb; ++kb)
                                tma_prefetch_3d(&tmap_k, kBoxCols * kb, t.h, static_cast<int>(t.row0));
                        walk_advance(p, w, p.pair_ds, p.pair_dh);
                    }
                } else if (q + 1 < n_local) {
                    walk_advance(p, w, p.pair_ds, p.pair_dh);
                }
                const uint32_t loads = __ballot_sync(0xFu, !pf_lane && t.L > 0) & 3u;
#pragma unroll
                for (kc = 0; kc < nkc; ++kc) {
                    const int64_t v = q * nkc + kc;
                    const int nb = kF32Keys ? 1 : ((2 * kc + 1 < nkb) ? 2 : 1);
                    const int box0 = kF32Keys ? kc : 2 * kc;
                    const int s = static_cast<int>(v % kNumStages);
                    const uint32_t ph = static_cast<uint32_t>((v / kNumStages) & 1);
                    const uint32_t st = sbase + kOffK + s * kUnitBytes;
                    int ok = 1;
                    if (lane == 0) {
                        ok = mbar_wait(bar_empty + 8 * s, ph ^ 1) ? 1 : 0;
                        if (!ok) record_timeout(p, abort_flag);
                        else mbar_arrive_expect_tx(bar_full + 8 * s, __popc(loads) * nb * kBoxBytes);
                    }
                    if (!__shfl_sync(0xFu, ok, 0)) {
                        failed = true;
                        break;
                    }
                    if (!pf_lane && t.L > 0)
#pragma unroll
                        for (int kh = 0; kh < nb; ++kh)
                            tma_load_3d(st + (2 * kh + tt) * kBoxBytes, &tmap_k, bar_full + 8 * s,
                                        kBoxCols * (box0 + kh), t.h, static_cast<int>(t.row0));
                }
                if (failed) break;
            }
            const int64_t v = q * nkc + (failed ? kc : 0);   // units issued
            if (lane == 0) {
                // Drain: every issued load has landed and every stage's MMAs committed.
                const int64_t first = v > kNumStages ? v - kNumStages : 0;
                for (int64_t r = first; r < v; ++r) {
                    const int s = static_cast<int>(r % kNumStages);
                    const uint32_t ph = static_cast<uint32_t>((r / kNumStages) & 1);
                    if (!mbar_wait(bar_full + 8 * s, ph)) record_timeout(p, abort_flag);
                    if (!mbar_wait(bar_empty + 8 * s, ph)) record_timeout(p, abort_flag);
                }
            }
        }
    } else if (kF32Keys && warp >= kCvtWarp0) {
        // The converter warps split every key unit v.  Each key x becomes
        // big = x rounded to tf32 (split_tf32), written back in place for the
        // kind::tf32 product big big^T, and small = x - big; bf16(big) and
        // bf16(small) go to pair unit v % kNumRem (once the MMAs that read its
        // previous contents have completed) as one 128-row operand whose
        // 128-byte rows hold [bf16(big) of the unit's 32 columns | bf16(small)
        // of them], for the cross products big small^T + small big^T on the
        // kind::f16 path.  Then the warp signals the unit's converted barrier.
        const int64_t units = n_local * nkc;
        // Work items: (row r of the unit's 128, column octet o of 4), eight
        // consecutive rows per warp instruction (conflict-free in the 128-byte
        // swizzle).
        constexpr int kItems = 128 * 4 / (32 * L::kCvtPerGroup);   // per lane
        const int cg = (warp - kCvtWarp0) / L::kCvtPerGroup;       // converter group
        const int t0 = ((warp - kCvtWarp0) % L::kCvtPerGroup) * 32 + lane;
        for (int64_t v = cg; v < units; v += L::kCvtGroups) {
            if (*abort_flag) break;
            const int s = static_cast<int>(v % kNumStages);
            const uint32_t ph = static_cast<uint32_t>((v / kNumStages) & 1);
            const int u = static_cast<int>(v % kRemMod);
            const uint32_t phr = static_cast<uint32_t>((v / kRemMod) & 1);
            int ok = 1;
            if (lane == 0)
                ok = (mbar_wait(bar_full + 8 * s, ph) && mbar_wait(bar_rfree + 8 * u, phr ^ 1)) ? 1 : 0;
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
                if (lane == 0) record_timeout(p, abort_flag);
                break;
            }
            uint8_t *const ku = smem + kOffK + s * kUnitBytes;
            uint8_t *const pu = smem + L::kOffRem + u * L::kRemBytes;
            // The lane's items go in batches whose loads are all issued before
            // the batch's first store (the pair unit is not known not to alias
            // the key unit, so a load left behind a store would wait for it).
            constexpr int kBatch = kItems < 4 ? kItems : 4;
#pragma unroll
            for (int b0 = 0; b0 < kItems; b0 += kBatch) {
                float4 xa[kBatch], xb[kBatch];
#pragma unroll
                for (int it = 0; it < kBatch; ++it) {
                    const int item = t0 + 32 * L::kCvtPerGroup * (b0 + it);
                    const int r = item >> 2, o = item & 3;
                    xa[it] = *reinterpret_cast<const float4 *>(ku + r * 128 + (((2 * o) ^ (r & 7)) << 4));
                    xb[it] = *reinterpret_cast<const float4 *>(ku + r * 128 + (((2 * o + 1) ^ (r & 7)) << 4));
                }
#pragma unroll
                for (int it = 0; it < kBatch; ++it) {
                    const int item = t0 + 32 * L::kCvtPerGroup * (b0 + it);
                    const int r = item >> 2, o = item & 3;
                    const float xv[8] = {xa[it].x, xa[it].y, xa[it].z, xa[it].w,
                                         xb[it].x, xb[it].y, xb[it].z, xb[it].w};
                    uint32_t bg[8], sm[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) split_tf32(xv[e], bg[e], sm[e]);
                    *reinterpret_cast<uint4 *>(ku + r * 128 + (((2 * o) ^ (r & 7)) << 4)) =
                        make_uint4(bg[0], bg[1], bg[2], bg[3]);
                    *reinterpret_cast<uint4 *>(ku + r * 128 + (((2 * o + 1) ^ (r & 7)) << 4)) =
                        make_uint4(bg[4], bg[5], bg[6], bg[7]);
                    uint32_t pb[4], ps[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pb[e] = pack16x2<kOutBF16>(__uint_as_float(bg[2 * e]), __uint_as_float(bg[2 * e + 1]));
                        ps[e] = pack16x2<kOutBF16>(__uint_as_float(sm[2 * e]), __uint_as_float(sm[2 * e + 1]));
                    }
                    *reinterpret_cast<uint4 *>(pu + r * 128 + ((o ^ (r & 7)) << 4)) =
                        make_uint4(pb[0], pb[1], pb[2], pb[3]);
                    *reinterpret_cast<uint4 *>(pu + r * 128 + (((4 + o) ^ (r & 7)) << 4)) =
                        make_uint4(ps[0], ps[1], ps[2], ps[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_cvt + 8 * u);
        }
    } else if (kF32Keys && warp == kMmaWarp) {
        // Lane 0 waits for the converted unit and issues per K step of 8 the
        // tf32 product big big^T, and per K step of 16 the two bf16 cross
        // products from the pair unit (A and B descriptors 64 bytes apart in
        // its rows); their completion frees both the key unit and the pair unit.
        if (lane == 0) {
            int64_t q = 0;
            bool failed = false;
            for (; q < n_local; ++q) {
                if (*abort_flag) break;
                const int w = static_cast<int>(q % kNumWG);
                const uint32_t phw = static_cast<uint32_t>((q / kNumWG) & 1);
                const uint32_t d = tmem_base + static_cast<uint32_t>(128 * w);
                for (int kc = 0; kc < nkc; ++kc) {
                    const int64_t v = q * nkc + kc;
                    const int s = static_cast<int>(v % kNumStages);
                    const int u = static_cast<int>(v % kRemMod);
                    const uint32_t phr = static_cast<uint32_t>((v / kRemMod) & 1);
                    if (!mbar_wait(bar_cvt + 8 * u, phr) ||
                        (kc == 0 && !mbar_wait(bar_tempty + 8 * w, phw ^ 1))) {
                        record_timeout(p, abort_flag);
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = sbase + kOffK + s * kUnitBytes;
                    const uint32_t sp = sbase + L::kOffRem + u * L::kRemBytes;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t db = smem_desc_sw128(st + ks * 32);
                        tc_mma_tf32(d, db, db, p.idesc, (kc | ks) ? 1u : 0u);
                    }
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t pb = smem_desc_sw128(sp + ks * 32), ps = smem_desc_sw128(sp + 64 + ks * 32);
                        tc_mma_f16(d, pb, ps, kIdescBf16, 1u);
                        tc_mma_f16(d, ps, pb, kIdescBf16, 1u);
                    }
                    tc_commit(bar_empty + 8 * s);
                    tc_commit(bar_rfree + 8 * u);
                    if (kc == nkc - 1) tc_commit(bar_tfull + 8 * w);
                }
                if (failed) break;
            }
            if (q > 0) {
                const int64_t r = q - 1;
                const int w = static_cast<int>(r % kNumWG);
                if (!mbar_wait(bar_tfull + 8 * w, static_cast<uint32_t>((r / kNumWG) & 1)))
                    record_timeout(p, abort_flag);
            }
        }
    } else if (warp == kMmaWarp) {
        if (kUseTmem && lane == 0) {
            int64_t q = 0;          // ends as the number of pairs whose Gram was committed
            bool failed = false;
            for (; q < n_local; ++q) {
                if (*abort_flag) break;
                const int w = static_cast<int>(q % kNumWG);
                const uint32_t phw = static_cast<uint32_t>((q / kNumWG) & 1);
                const uint32_t d = tmem_base + static_cast<uint32_t>(128 * w);
#pragma unroll
                for (int kc = 0; kc < nkc; ++kc) {
                    const int64_t v = q * nkc + kc;
                    const int s = static_cast<int>(v % kNumStages);
                    const uint32_t ph = static_cast<uint32_t>((v / kNumStages) & 1);
                    if (!mbar_wait(bar_full + 8 * s, ph) ||
                        (kc == 0 && !mbar_wait(bar_tempty + 8 * w, phw ^ 1))) {
                        record_timeout(p, abort_flag);
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    // One N = 128 product per K step: rows and columns both run over
                    // the pair's 128 key rows; each tile reads its own diagonal block.
                    const uint32_t st = sbase + kOffK + s * kUnitBytes;
                    const int nb = (2 * kc + 1 < nkb) ? 2 : 1;
#pragma unroll
                    for (int kh = 0; kh < nb; ++kh) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t a_addr = st + kh * 2 * kBoxBytes + ks * 32;
                            if constexpr (kTf32Gram)
                                tc_mma_tf32(d, smem_desc_sw128(a_addr), smem_desc_sw128(a_addr), p.idesc,
                                            (kc | kh | ks) ? 1u : 0u);
                            else
                                tc_mma_f16(d, smem_desc_sw128(a_addr), smem_desc_sw128(a_addr), p.idesc,
                                           (kc | kh | ks) ? 1u : 0u);
                        }
                    }
                    tc_commit(bar_empty + 8 * s);
                    if (kc == nkc - 1) tc_commit(bar_tfull + 8 * w);
                }
                if (failed) break;
            }
            // The last pair's MMAs must be complete before TMEM is released.
            if (q > 0) {
                const int64_t r = q - 1;
                const int w = static_cast<int>(r % kNumWG);
                if (!mbar_wait(bar_tfull + 8 * w, static_cast<uint32_t>((r / kNumWG) & 1)))
                    record_timeout(p, abort_flag);
            }
        }
    } else {
        // ------------------------------------------------ consumer warpgroups
        const int wg = warp >> 2;
        const int qd = warp & 3;                 // TMEM lane quadrant of this warp
        const int tt_e = qd >> 1;                // epilogue: tile of this thread's row
        const int i_e = 32 * (qd & 1) + lane;    // epilogue: row within the tile
        const int tid = threadIdx.x & 127;       // thread index inside the warpgroup
        const int g8 = lane >> 2, t4 = lane & 3; // mma.sync fragment coordinates
        uint8_t *abuf = smem + L::kOffA + wg * kAWGBytes;
        float *const At0 = reinterpret_cast<float *>(abuf);
        float *const At1 = reinterpret_cast<float *>(abuf + kATile1Off);
        auto At = [At0, At1](int t) { return t ? At1 : At0; };
        float *gbuf = reinterpret_cast<float *>(smem + L::kOffG + wg * kGWGBytes);   // [parity][tile][64]
        float *vbuf = gbuf + 2 * 2 * kChunk;                                       // [parity][tile][64]
        const int bar_id = 1 + wg;

        int64_t q = wg;
        // This thread's tile (tt_e) of each of the warpgroup's pairs.
        TileWalk wk = walk_init(p, static_cast<uint32_t>(2 * (blockIdx.x + q * gridDim.x) + tt_e));
        Tile cur = walk_tile(p, wk);
        RowIn rin = load_row(p, cur, i_e);

        for (int r = 0; q < n_local; ++r, q += kNumWG) {
            // Prefetch the next pair's schedule and row inputs.
            const int64_t qn = q + kNumWG;
            Tile nx;
            nx.L = 0;
            nx.row0 = 0;
            nx.h = 0;
            if (qn < n_local) {
                walk_advance(p, wk, p.wg_ds, p.wg_dh);
                nx = walk_tile(p, wk);
            }
            const RowIn rnext = load_row(p, nx, i_e);

            if ((qd & 1) == 0 && lane == 0) bulk_wait_read();   // this warp's previous store
            // The warpgroup's input: its Gram in TMEM, or in the solve mode its A
            // tiles in stage wg (pair q = wg + 3r uses stage q % 3 = wg).
            const uint32_t bar_in = kUseTmem ? bar_tfull + 8 * wg : bar_full + 8 * wg;
            if (qd == 3 && lane == 0) {
                int ok = mbar_wait(bar_in, static_cast<uint32_t>(r & 1)) ? 1 : 0;
                if (!ok) record_timeout(p, abort_flag);
                wg_flag[wg] = ok;
            }
            // Gate factors around the chunk's reference: exp(g_i - g_j) =
            // u_i * v_j with u_i = exp(g_i - gref), v_j = exp(gref - g_j).  Used
            // only when every |g - gref| <= 30 in both tiles (no overflow, and
            // the [-50, 50] clamp cannot bind); otherwise the clamped
            // exp(g_i - g_j) is evaluated directly.
            const Tile te = cur;
            const bool rowok = i_e < te.L;
            float ui = 1.0f, vi = 1.0f;
            bool unsafe = false;
            if (MODE != kModeSolve && p.g && rowok) {
                const float d = rin.g - 0.5f * (rin.gfirst + rin.glast);
                unsafe = !(fabsf(d) <= 30.0f);
                ui = expf(d);
                vi = expf(-d);
            }
            float *gcur = gbuf + (r & 1) * 2 * kChunk + tt_e * kChunk;
            float *vcur = vbuf + (r & 1) * 2 * kChunk + tt_e * kChunk;
            gcur[i_e] = rin.g;
            vcur[i_e] = rowok ? vi : 0.0f;
            const bool direct = named_bar_red_or(bar_id, 128, unsafe);   // B2: g, v ready; A free
            if (!wg_flag[wg]) break;
            if constexpr (kUseTmem) tc_fence_after();

            // ---- epilogue: S row from TMEM -> A row in shared memory (in the kkt
            //      mode: into the fp32 staging, masked to the strict lower part);
            //      solve mode: A row from the stage -> shared memory
            if constexpr (MODE == kModeSolve) {
                // Every thread acquires the stage's completed phase itself.
                if (!mbar_wait(bar_in, static_cast<uint32_t>(r & 1))) record_timeout(p, abort_flag);
                static_assert(MODE != kModeSolve || kNumStages == kNumWG, "stage wg holds pair q's A tiles");
                const uint8_t *sa = smem + kOffK + wg * kUnitBytes + tt_e * kBoxBytes + i_e * 128;
                float4 *Arow = reinterpret_cast<float4 *>(At(tt_e) + a_row<kP>(i_e));
                const int n4 = (qd & 1) ? 16 : 8;
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4) {
                    if (j4 < n4) {
                        const float4 v = *reinterpret_cast<const float4 *>(
                            sa + (j4 >> 3) * 2 * kBoxBytes + (((j4 & 7) ^ (i_e & 7)) << 4));
                        Arow[j4] = rowok ? v : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * wg);
            } else
            {
                uint32_t sr[64];
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * qd) << 16) +
                                       static_cast<uint32_t>(128 * wg + 64 * tt_e);
                {
                    uint32_t (&lo)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[0]);
                    uint32_t (&hi)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[32]);
                    tmem_ld32(taddr, lo);
                    tmem_ld32(taddr + 32, hi);
                }
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 64; ++j) reg_fence(sr[j]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty + 8 * wg);

                float4 *Arow = reinterpret_cast<float4 *>(At(tt_e) + a_row<kP>(i_e));
                // Row i of block I = i / 16 only needs columns j < 16 (I + 1): the
                // blocks left of the diagonal and the diagonal block itself (A is
                // strictly lower).  The kkt mode writes whole rows, zero at and
                // above the diagonal.
                const int n4 = MODE == kModeKkt ? 16 : 4 * ((i_e >> 4) + 1);
                uint8_t *const sk = abuf + (tt_e ? kStage1Off : 0);
                auto put = [&](int j4, float4 a) {
                    if constexpr (MODE == kModeKkt) {
                        const int j = 4 * j4;
                        a.x = j + 0 < i_e ? a.x : 0.0f;
                        a.y = j + 1 < i_e ? a.y : 0.0f;
                        a.z = j + 2 < i_e ? a.z : 0.0f;
                        a.w = j + 3 < i_e ? a.w : 0.0f;
                        *reinterpret_cast<float4 *>(sk + stage_piece_off<false>(i_e, j4)) = a;
                    } else {
                        Arow[j4] = a;
                    }
                };
                if (!rowok) {
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4)
                        if (j4 < n4) put(j4, z);
                } else if (!direct) {
                    const float w = beta_value(p, rin.beta) * ui;
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        if (j4 < n4) {
                            const float4 v = reinterpret_cast<const float4 *>(vcur)[j4];
                            float4 a;
                            a.x = (__uint_as_float(sr[4 * j4 + 0]) * w) * v.x;
                            a.y = (__uint_as_float(sr[4 * j4 + 1]) * w) * v.y;
                            a.z = (__uint_as_float(sr[4 * j4 + 2]) * w) * v.z;
                            a.w = (__uint_as_float(sr[4 * j4 + 3]) * w) * v.w;
                            put(j4, a);
                        }
                    }
                } else {
                    const float gi = rin.g, bi = beta_value(p, rin.beta);
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        if (j4 < n4) {
                            const float4 gj = reinterpret_cast<const float4 *>(gcur)[j4];
                            float4 a;
                            a.x = bi * __uint_as_float(sr[4 * j4 + 0]) *
                                  __expf(fminf(fmaxf(gi - gj.x, -50.f), 50.f));
                            a.y = bi * __uint_as_float(sr[4 * j4 + 1]) *
                                  __expf(fminf(fmaxf(gi - gj.y, -50.f), 50.f));
                            a.z = bi * __uint_as_float(sr[4 * j4 + 2]) *
                                  __expf(fminf(fmaxf(gi - gj.z, -50.f), 50.f));
                            a.w = bi * __uint_as_float(sr[4 * j4 + 3]) *
                                  __expf(fminf(fmaxf(gi - gj.w, -50.f), 50.f));
                            put(j4, a);
                        }
                    }
                }
            }
            // The kkt mode is done: its rows are in the staging.
            if constexpr (MODE != kModeKkt) {
                // The diagonal blocks this warp inverts below are exactly the 32 rows it
                // has just written (tile qd >> 1, rows 32 (qd & 1) ..), so a warp-level
                // barrier is enough here.
                __syncwarp();

                // ---- diagonal inverses: thread -> (tile, block I, row c)
                const int dt = tid >> 6, dI = (tid >> 4) & 3, dc = tid & 15;
                float drow[16];
                diag_inverse_row<kP>(At(dt) + a_row<kP>(16 * dI) + 16 * dI, dc, drow);
                {
                    float4 *dst = reinterpret_cast<float4 *>(At(dt) + a_row<kP>(16 * dslot_r(dI) + dc) +
                                                             16 * dslot_c(dI));
    #pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        dst[j4] = make_float4(drow[4 * j4], drow[4 * j4 + 1], drow[4 * j4 + 2], drow[4 * j4 + 3]);
                }
                named_bar_sync(bar_id, 128);                       // B3b: D blocks ready

                // ---- off-diagonal blocks on tensor cores: warp -> (tile, block column);
                //      then X rows are assembled in the A buffer (after B4 in both branches)
                const int mt = qd & 1;
                uint8_t *const st_m = abuf + (mt ? kStage1Off : 0);
                if (qd < 2) {
                    float z0[3][2][4];
                    merge_column<0, OUT != kOutBF16, kP>(At(mt), g8, t4, z0);
                    named_bar_sync(bar_id, 128);                   // B4: A and D no longer read
                    stage_block_T<OUT>(st_m, 1, 0, z0[0], g8, t4);
                    stage_block_T<OUT>(st_m, 2, 0, z0[1], g8, t4);
                    stage_block_T<OUT>(st_m, 3, 0, z0[2], g8, t4);
                } else {
                    float z1[2][2][4], z2[1][2][4];
                    merge_column<1, OUT != kOutBF16, kP>(At(mt), g8, t4, z1);
                    merge_column<2, OUT != kOutBF16, kP>(At(mt), g8, t4, z2);
                    named_bar_sync(bar_id, 128);                   // B4: A and D no longer read
                    stage_block_T<OUT>(st_m, 2, 1, z1[0], g8, t4);
                    stage_block_T<OUT>(st_m, 3, 1, z1[1], g8, t4);
                    stage_block_T<OUT>(st_m, 3, 2, z2[0], g8, t4);
                }
                {
                    const float4 dv[4] = {make_float4(drow[0], drow[1], drow[2], drow[3]),
                                          make_float4(drow[4], drow[5], drow[6], drow[7]),
                                          make_float4(drow[8], drow[9], drow[10], drow[11]),
                                          make_float4(drow[12], drow[13], drow[14], drow[15])};
                    stage_diag_row<OUT>(abuf + (dt ? kStage1Off : 0), 16 * dI + dc, dI, dv);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(bar_id, 128);                       // B5: X complete

            // ---- store: full chunks by TMA from the staging, partial chunks row by row
            // Lane 0 of warps 0 and 2 stores the tile its warp's rows belong to.
            if (lane == 0 && (qd & 1) == 0 && cur.L == kChunk) {
                const uint32_t src = smem_u32(abuf + (tt_e ? kStage1Off : 0));
                tma_store_3d(&tmap_out, src, 0, cur.h, static_cast<int>(cur.row0));
                if (OUT == kOutF32) tma_store_3d(&tmap_out, src + 8192, 32, cur.h, static_cast<int>(cur.row0));
                bulk_commit();
            }
            {
                const int st_t = tt_e;
                const Tile ts = cur;
                if (ts.L > 0 && ts.L < kChunk) {
                    const uint8_t *sb = abuf + (st_t ? kStage1Off : 0);
                    constexpr int kPieces = OUT != kOutF32 ? 8 : 16;
                    constexpr int kRowsPerIt = 32 / kPieces;
#pragma unroll 2
                    for (int it = 0; it < 32 / kRowsPerIt; ++it) {
                        const int rr = 32 * (qd & 1) + kRowsPerIt * it + lane / kPieces;
                        const int piece = lane % kPieces;
                        if (rr < ts.L) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(sb + stage_piece_off<OUT != kOutF32>(rr, piece));
                            const int64_t orow = (ts.row0 + rr) * p.H + ts.h;
                            *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) +
                                                       orow * (OUT != kOutF32 ? 128 : 256) + 16 * piece) = v;
                        }
                    }
                }
            }
            cur = nx;
            rin = rnext;
        }
        if (lane == 0 && (qd & 1) == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (kUseTmem && warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------------------ chunk 128
// (I + A)^{-1} of 128-token chunks (the chunk of the PyPTO page
// "GatedDeltaRule算子性能优化案例", section 3.2: TileShape [128, 128]; its
// section 3.3.2 inverts the tile through 8 blocks of 16 x 16).  A chunk is one
// pipeline pair whose two "tiles" are its halves, so the producer, the stage
// ring and the M = N = 128 Gram are those of the 64-token kernel, and TMEM now
// holds all of S, including the cross block S21 (second-half rows, first-half
// columns).  With the halves' inverses X11 = (I + A11)^{-1} and
// X22 = (I + A22)^{-1} (the 64-token solve on each half),
//     X = [[X11, 0], [X21, X22]],   X21 = -X22 A21 X11,
// and X21 comes from two more block products on the tensor cores.  Three
// consumer warpgroups (128 rows each) on a two-stage key ring; per warpgroup
// three 64 x 64 fp32 matrices: M0 = A11 then X11, M1 = A22 then X22, M2 = A21
// then X21.
constexpr int kC128WG = 3;
constexpr int kC128Stages = 2;
constexpr int kC128Producer = 4 * kC128WG;
constexpr int kC128Mma = 4 * kC128WG + 1;
constexpr int kC128Threads = 32 * (4 * kC128WG + 2);
constexpr int kC128Pitch = 68;                             // matrix rows 68 floats apart
constexpr int kMatBytes = kChunk * kC128Pitch * 4;        // 17408
constexpr int kC128M1Off = kMatBytes + 16;                // other banks than M0
constexpr int kC128M2Off = 2 * kMatBytes + 32;
constexpr int kC128WGBytes = kC128M2Off + kMatBytes;       // 52256 (16-byte aligned matrices)
constexpr int kC128GBytes = 2 * 2 * 128 * 4;              // g and v of 128 rows, double buffered
constexpr int kC128OffA = kOffK + kC128Stages * kStageBytes;
constexpr int kC128OffG = kC128OffA + kC128WG * kC128WGBytes;
constexpr int kC128OffBar = kC128OffG + kC128WG * kC128GBytes;
constexpr int kC128OffMisc = kC128OffBar + (2 * kC128Stages + 2 * kC128WG) * 8;
constexpr int kC128SmemBytes = kC128OffMisc + 64 + 1024;
constexpr uint32_t kC128TmemCols = 512;
static_assert(kC128WGBytes % 16 == 0, "chunk-128 matrices");
// 16-bit output of a full chunk leaves by four TMA stores of 64 x 64 boxes
// (X11, the zero block, X21, X22), staged 128-byte swizzled at the first
// 1024-byte boundary of the warpgroup's matrices: over M0 and most of M1 (read
// into registers first), never over M2.
__host__ __device__ constexpr int c128_stage_off(int wg) {
    return (1024 - (kC128OffA + wg * kC128WGBytes) % 1024) % 1024;
}
static_assert(c128_stage_off(0) + 4 * 8192 <= kC128M2Off && c128_stage_off(1) + 4 * 8192 <= kC128M2Off &&
                  c128_stage_off(2) + 4 * 8192 <= kC128M2Off,
              "chunk-128 staging stays clear of M2");
static_assert(kC128SmemBytes <= 232448, "chunk-128 shared memory budget");

// Piece q (columns 8q .. 8q + 7) of row r of a lower-triangular 64 x 64 block
// (fp32 rows kC128Pitch apart), above-diagonal values as zeros, packed to the
// 16-bit output type.
template <int OUT>
__device__ __forceinline__ void c128_piece_lower(const float *M, int r, int q, uint32_t (&w)[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(M + r * kC128Pitch + 8 * q);
    const float4 b = *reinterpret_cast<const float4 *>(M + r * kC128Pitch + 8 * q + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float m[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = 8 * q + e <= r ? v[e] : 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = pack16x2<OUT>(m[2 * e], m[2 * e + 1]);
}

// The half tt (0 or 1) of a 128-token chunk as a 64-row tile.
__device__ __forceinline__ Tile half_of(const Tile &c, int tt) {
    Tile t;
    t.h = c.h;
    t.row0 = c.row0 + 64 * tt;
    const int l = c.L - 64 * tt;
    t.L = l < 0 ? 0 : (l > 64 ? 64 : l);
    return t;
}

template <int OUT, int NKB>
__global__ void __launch_bounds__(kC128Threads, 1)
    kkt_solve_c128_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_out, const Params p) {
    constexpr bool SPLIT = OUT != kOutBF16;
    constexpr bool kTmaOut = OUT != kOutF32;     // 16-bit output: full chunks by TMA store
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + kC128OffBar;                   // [kC128Stages]
    const uint32_t bar_empty = bar_full + 8 * kC128Stages;            // [kC128Stages]
    const uint32_t bar_tfull = bar_empty + 8 * kC128Stages;           // [kC128WG]
    const uint32_t bar_tempty = bar_tfull + 8 * kC128WG;             // [kC128WG]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kC128OffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kC128OffMisc + 4);
    volatile int *wg_flag = reinterpret_cast<volatile int *>(smem + kC128OffMisc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kC128Stages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int w = 0; w < kC128WG; ++w) {
            mbar_init(bar_tfull + 8 * w, 1);
            mbar_init(bar_tempty + 8 * w, 4);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kC128Mma) {
        tmem_alloc(smem_u32(tmem_slot), kC128TmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    const int64_t n_local = (p.n_pairs > blockIdx.x)
                                ? (p.n_pairs - 1 - blockIdx.x) / gridDim.x + 1
                                : 0;
    constexpr int nkb = NKB;
    constexpr int nkc = (nkb + 1) >> 1;
    constexpr int kPrefetchPairs = 0;        // see prefetch_pairs

    if (warp == kC128Producer) {
        // As in the 64-token kernel; lane tt & 1 issues the copies of half tt.
        if (lane < 4) {
            if (lane == 0)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k))
                             : "memory");
            const int tt = lane & 1;
            const bool pf_lane = lane >= 2;
            TileWalk w = walk_init<128>(p, static_cast<uint32_t>(blockIdx.x));
            if (pf_lane)
                for (int i = 0; i < kPrefetchPairs; ++i) walk_advance<128>(p, w, p.pair_ds, p.pair_dh);
            int64_t q = 0;
            int kc = 0;
            bool failed = false;
            for (; q < n_local; ++q) {
                int stop = (lane == 0) ? *abort_flag : 0;
                if (__shfl_sync(0xFu, stop, 0)) break;
                const Tile t = half_of(walk_tile<128>(p, w), tt);
                if (pf_lane) {
                    if (q + kPrefetchPairs < n_local) {
                        if (t.L > 0)
#pragma unroll
                            for (int kb = 0; kb < nkb; ++kb)
                                tma_prefetch_3d(&tmap_k, 64 * kb, t.h, static_cast<int>(t.row0));
                        walk_advance<128>(p, w, p.pair_ds, p.pair_dh);
                    }
                } else if (q + 1 < n_local) {
                    walk_advance<128>(p, w, p.pair_ds, p.pair_dh);
                }
                const uint32_t loads = __ballot_sync(0xFu, !pf_lane && t.L > 0) & 3u;
#pragma unroll
                for (kc = 0; kc < nkc; ++kc) {
                    const int64_t v = q * nkc + kc;
                    const int nb = (2 * kc + 1 < nkb) ? 2 : 1;
                    const int s = static_cast<int>(v % kC128Stages);
                    const uint32_t ph = static_cast<uint32_t>((v / kC128Stages) & 1);
                    const uint32_t st = sbase + kOffK + s * kStageBytes;
                    int ok = 1;
                    if (lane == 0) {
                        ok = mbar_wait(bar_empty + 8 * s, ph ^ 1) ? 1 : 0;
                        if (!ok) record_timeout(p, abort_flag);
                        else mbar_arrive_expect_tx(bar_full + 8 * s, __popc(loads) * nb * kBoxBytes);
                    }
                    if (!__shfl_sync(0xFu, ok, 0)) {
                        failed = true;
                        break;
                    }
                    if (!pf_lane && t.L > 0)
#pragma unroll
                        for (int kh = 0; kh < nb; ++kh)
                            tma_load_3d(st + (2 * kh + tt) * kBoxBytes, &tmap_k, bar_full + 8 * s,
                                        64 * (2 * kc + kh), t.h, static_cast<int>(t.row0));
                }
                if (failed) break;
            }
            const int64_t v = q * nkc + (failed ? kc : 0);
            if (lane == 0) {
                const int64_t first = v > kC128Stages ? v - kC128Stages : 0;
                for (int64_t r = first; r < v; ++r) {
                    const int s = static_cast<int>(r % kC128Stages);
                    const uint32_t ph = static_cast<uint32_t>((r / kC128Stages) & 1);
                    if (!mbar_wait(bar_full + 8 * s, ph)) record_timeout(p, abort_flag);
                    if (!mbar_wait(bar_empty + 8 * s, ph)) record_timeout(p, abort_flag);
                }
            }
        }
    } else if (warp == kC128Mma) {
        if (lane == 0) {
            int64_t q = 0;
            bool failed = false;
            for (; q < n_local; ++q) {
                if (*abort_flag) break;
                const int w = static_cast<int>(q % kC128WG);
                const uint32_t phw = static_cast<uint32_t>((q / kC128WG) & 1);
                const uint32_t d = tmem_base + static_cast<uint32_t>(128 * w);
#pragma unroll
                for (int kc = 0; kc < nkc; ++kc) {
                    const int64_t v = q * nkc + kc;
                    const int s = static_cast<int>(v % kC128Stages);
                    const uint32_t ph = static_cast<uint32_t>((v / kC128Stages) & 1);
                    if (!mbar_wait(bar_full + 8 * s, ph) ||
                        (kc == 0 && !mbar_wait(bar_tempty + 8 * w, phw ^ 1))) {
                        record_timeout(p, abort_flag);
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = sbase + kOffK + s * kStageBytes;
                    const int nb = (2 * kc + 1 < nkb) ? 2 : 1;
#pragma unroll
                    for (int kh = 0; kh < nb; ++kh) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint32_t a_addr = st + kh * 2 * kBoxBytes + ks * 32;
                            tc_mma_f16(d, smem_desc_sw128(a_addr), smem_desc_sw128(a_addr), p.idesc,
                                       (kc | kh | ks) ? 1u : 0u);
                        }
                    }
                    tc_commit(bar_empty + 8 * s);
                    if (kc == nkc - 1) tc_commit(bar_tfull + 8 * w);
                }
                if (failed) break;
            }
            if (q > 0) {
                const int64_t r = q - 1;
                const int w = static_cast<int>(r % kC128WG);
                if (!mbar_wait(bar_tfull + 8 * w, static_cast<uint32_t>((r / kC128WG) & 1)))
                    record_timeout(p, abort_flag);
            }
        }
    } else {
        // ------------------------------------------------ consumer warpgroups
        const int wg = warp >> 2;
        const int qd = warp & 3;
        const int i = 32 * qd + lane;            // row of the chunk = TMEM lane
        const int hf = qd >> 1;                  // half of this row
        const int ih = i & 63;                   // row within the half
        const int tid = threadIdx.x & 127;
        const int g8 = lane >> 2, t4 = lane & 3;
        uint8_t *mb = smem + kC128OffA + wg * kC128WGBytes;
        float *const M0 = reinterpret_cast<float *>(mb);
        float *const M1 = reinterpret_cast<float *>(mb + kC128M1Off);
        float *const M2 = reinterpret_cast<float *>(mb + kC128M2Off);
        auto Mh = [M0, M1](int t) { return t ? M1 : M0; };
        auto blk = [](float *M, int I, int J) { return M + 16 * I * kC128Pitch + 16 * J; };
        float *gbuf = reinterpret_cast<float *>(smem + kC128OffG + wg * kC128GBytes);   // [parity][128]
        float *vbuf = gbuf + 2 * 128;
        const int bar_id = 1 + wg;

        int64_t q = wg;
        TileWalk wk = walk_init<128>(p, static_cast<uint32_t>(blockIdx.x + q * gridDim.x));
        Tile cur = walk_tile<128>(p, wk);
        RowIn rin = load_row(p, cur, i);

        for (int r = 0; q < n_local; ++r, q += kC128WG) {
            const int64_t qn = q + kC128WG;
            Tile nx;
            nx.L = 0;
            nx.row0 = 0;
            nx.h = 0;
            if (qn < n_local) {
                walk_advance<128>(p, wk, p.wg_ds, p.wg_dh);
                nx = walk_tile<128>(p, wk);
            }
            const RowIn rnext = load_row(p, nx, i);

            // The previous chunk's TMA store has read its staging (over M0, M1)
            // before the barrier below lets the epilogue write the matrices.
            if (kTmaOut && tid == 0) bulk_wait_read();
            if (qd == 3 && lane == 0) {
                int ok = mbar_wait(bar_tfull + 8 * wg, static_cast<uint32_t>(r & 1)) ? 1 : 0;
                if (!ok) record_timeout(p, abort_flag);
                wg_flag[wg] = ok;
            }
            // Gate factors around the whole chunk's reference (the cross block
            // needs one reference for both halves); same safety rule as for 64.
            const bool rowok = i < cur.L;
            float ui = 1.0f, vi = 1.0f;
            bool unsafe = false;
            if (p.g && rowok) {
                const float dg = rin.g - 0.5f * (rin.gfirst + rin.glast);
                unsafe = !(fabsf(dg) <= 30.0f);
                ui = expf(dg);
                vi = expf(-dg);
            }
            float *gcur = gbuf + (r & 1) * 128;
            float *vcur = vbuf + (r & 1) * 128;
            gcur[i] = rin.g;
            vcur[i] = rowok ? vi : 0.0f;
            const bool direct = named_bar_red_or(bar_id, 128, unsafe);   // g, v ready; matrices free
            if (!wg_flag[wg]) break;
            tc_fence_after();

            // ---- epilogue: the diagonal block row into M0 / M1 and, for second-half
            //      rows, the cross block row into M2
            {
                const float bi = beta_value(p, rin.beta);
                const float w = bi * ui;
                const float gi = rin.g;
                const int npass = hf ? 2 : 1;
                for (int pass = 0; pass < npass; ++pass) {
                    const int cb = pass == 0 ? 64 * hf : 0;        // TMEM columns = partner rows
                    float *const Arowf = (pass == 0 ? Mh(hf) : M2) + ih * kC128Pitch;
                    // Diagonal block rows 0..31 only need columns j < 32.
                    const int nh = (pass == 1 || (qd & 1)) ? 2 : 1;
                    for (int hh = 0; hh < nh; ++hh) {              // 32 columns at a time
                        uint32_t sr[32];
                        tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * qd) << 16) +
                                      static_cast<uint32_t>(128 * wg + cb + 32 * hh),
                                  sr);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) reg_fence(sr[j]);
                        float4 *Arow = reinterpret_cast<float4 *>(Arowf + 32 * hh);
                        const float4 *vj = reinterpret_cast<const float4 *>(vcur + cb + 32 * hh);
                        const float4 *gj = reinterpret_cast<const float4 *>(gcur + cb + 32 * hh);
                        if (!rowok) {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) Arow[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
                        } else if (!direct) {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 v = vj[j4];
                                float4 x;
                                x.x = (__uint_as_float(sr[4 * j4 + 0]) * w) * v.x;
                                x.y = (__uint_as_float(sr[4 * j4 + 1]) * w) * v.y;
                                x.z = (__uint_as_float(sr[4 * j4 + 2]) * w) * v.z;
                                x.w = (__uint_as_float(sr[4 * j4 + 3]) * w) * v.w;
                                Arow[j4] = x;
                            }
                        } else {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 gg = gj[j4];
                                float4 x;
                                x.x = bi * __uint_as_float(sr[4 * j4 + 0]) * __expf(fminf(fmaxf(gi - gg.x, -50.f), 50.f));
                                x.y = bi * __uint_as_float(sr[4 * j4 + 1]) * __expf(fminf(fmaxf(gi - gg.y, -50.f), 50.f));
                                x.z = bi * __uint_as_float(sr[4 * j4 + 2]) * __expf(fminf(fmaxf(gi - gg.z, -50.f), 50.f));
                                x.w = bi * __uint_as_float(sr[4 * j4 + 3]) * __expf(fminf(fmaxf(gi - gg.w, -50.f), 50.f));
                                Arow[j4] = x;
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_tempty + 8 * wg);
            }
            // A warp's diagonal blocks are the 32 rows it has just written.
            __syncwarp();

            // ---- diagonal inverses: thread -> (half, block, row) as in the 64 kernel
            const int dt = tid >> 6, dI = (tid >> 4) & 3, dc = tid & 15;
            float drow[16];
            diag_inverse_row<kC128Pitch>(Mh(dt) + 16 * dI * (kC128Pitch + 1), dc, drow);
            {
                float4 *dst = reinterpret_cast<float4 *>(Mh(dt) + (16 * dslot_r(dI) + dc) * kC128Pitch +
                                                         16 * dslot_c(dI));
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4)
                    dst[j4] = make_float4(drow[4 * j4], drow[4 * j4 + 1], drow[4 * j4 + 2], drow[4 * j4 + 3]);
            }
            named_bar_sync(bar_id, 128);                       // D blocks ready

            // ---- X11 and X22: the 64-token merge on each half, then written out as
            //      fp32 rows (diagonal blocks from the substitution rows)
            const int mt = qd & 1;
            if (qd < 2) {
                float z0[3][2][4];
                merge_column<0, SPLIT, kC128Pitch>(Mh(mt), g8, t4, z0);
                named_bar_sync(bar_id, 128);                   // A11, A22 no longer read
                store_block_T<kC128Pitch>(Mh(mt), 1, 0, z0[0], g8, t4);
                store_block_T<kC128Pitch>(Mh(mt), 2, 0, z0[1], g8, t4);
                store_block_T<kC128Pitch>(Mh(mt), 3, 0, z0[2], g8, t4);
            } else {
                float z1[2][2][4], z2[1][2][4];
                merge_column<1, SPLIT, kC128Pitch>(Mh(mt), g8, t4, z1);
                merge_column<2, SPLIT, kC128Pitch>(Mh(mt), g8, t4, z2);
                named_bar_sync(bar_id, 128);                   // A11, A22 no longer read
                store_block_T<kC128Pitch>(Mh(mt), 2, 1, z1[0], g8, t4);
                store_block_T<kC128Pitch>(Mh(mt), 3, 1, z1[1], g8, t4);
                store_block_T<kC128Pitch>(Mh(mt), 3, 2, z2[0], g8, t4);
            }
            {
                float4 *dst = reinterpret_cast<float4 *>(Mh(dt) + (16 * dI + dc) * kC128Pitch + 16 * dI);
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4)
                    dst[j4] = make_float4(drow[4 * j4], drow[4 * j4 + 1], drow[4 * j4 + 2], drow[4 * j4 + 3]);
            }
            named_bar_sync(bar_id, 128);                       // X11, X22 complete

            // ---- X21 = -X22 (A21 X11) in two balanced rounds, transposed as in the
            //      merge.  Round 1, warp -> block row M: P_MJ^T = sum_{K>=J}
            //      X11_KJ^T A21_MK^T for J = 0..3 (10 products), written as P_MJ
            //      over the warp's own A21 row of blocks.  Round 2, warp -> block
            //      column J: X21_IJ^T = -sum_{M<=I} P_MJ^T X22_IM^T (10 products).
            {
                const int M = qd;
                float pt[4][2][4];
#pragma unroll
                for (int J = 0; J < 4; ++J) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) pt[J][nt][e] = 0.0f;
#pragma unroll
                    for (int K2 = 0; K2 < 4; ++K2) {
                        if (K2 >= J) {
                            Frag16 f;
                            frag_from_dT<SPLIT, kC128Pitch>(blk(M0, K2, J), g8, t4, f);
                            mma3_times_blockT<SPLIT, kC128Pitch>(pt[J], f, blk(M2, M, K2), g8, t4);
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int J = 0; J < 4; ++J) store_block_T<kC128Pitch>(M2, M, J, pt[J], g8, t4);
            }
            named_bar_sync(bar_id, 128);                       // P complete
            {
                const int J = qd;
                float xt[4][2][4];
#pragma unroll
                for (int I = 0; I < 4; ++I) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) xt[I][nt][e] = 0.0f;
#pragma unroll
                    for (int M = 0; M < 4; ++M) {
                        if (M <= I) {
                            Frag16 f;
                            frag_from_dT<SPLIT, kC128Pitch>(blk(M2, M, J), g8, t4, f);
                            mma3_times_blockT<SPLIT, kC128Pitch>(xt[I], f, blk(M1, I, M), g8, t4);
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int I = 0; I < 4; ++I) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) xt[I][nt][e] = -xt[I][nt][e];
                    store_block_T<kC128Pitch>(M2, I, J, xt[I], g8, t4);
                }
            }
            named_bar_sync(bar_id, 128);                       // X complete

            // ---- store: every row of the chunk, 128 values; lower triangle of
            //      X11 / X22 (masked), X21 in full, zeros elsewhere.  A full chunk
            //      with 16-bit output goes out by TMA from the staging; otherwise
            //      row by row.
            if (kTmaOut && cur.L == 2 * kChunk) {
                uint8_t *const stg = mb + c128_stage_off(wg);
                // Item k of this thread: 16-byte piece q (8 values) of row r of a box.
                uint32_t x11[4][4], x22[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int idx = tid + 128 * k, r = idx >> 3, q = idx & 7;
                    c128_piece_lower<OUT>(M0, r, q, x11[k]);
                    c128_piece_lower<OUT>(M1, r, q, x22[k]);
                }
                named_bar_sync(bar_id, 128);                   // M0, M1 read: the staging may cover them
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int idx = tid + 128 * k, r = idx >> 3, q = idx & 7;
                    const uint32_t off = stage_piece_off<true>(r, q);
                    const float4 a = *reinterpret_cast<const float4 *>(M2 + r * kC128Pitch + 8 * q);
                    const float4 b = *reinterpret_cast<const float4 *>(M2 + r * kC128Pitch + 8 * q + 4);
                    *reinterpret_cast<uint4 *>(stg + off) = make_uint4(x11[k][0], x11[k][1], x11[k][2], x11[k][3]);
                    *reinterpret_cast<uint4 *>(stg + 8192 + off) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(stg + 16384 + off) =
                        make_uint4(pack16x2<OUT>(a.x, a.y), pack16x2<OUT>(a.z, a.w), pack16x2<OUT>(b.x, b.y),
                                   pack16x2<OUT>(b.z, b.w));
                    *reinterpret_cast<uint4 *>(stg + 24576 + off) = make_uint4(x22[k][0], x22[k][1], x22[k][2], x22[k][3]);
                }
                fence_proxy_async_smem();
                named_bar_sync(bar_id, 128);                   // staging complete
                if (tid == 0) {
                    const uint32_t src = smem_u32(stg);
                    const int row0 = static_cast<int>(cur.row0);
                    tma_store_3d(&tmap_out, src, 0, cur.h, row0);
                    tma_store_3d(&tmap_out, src + 8192, 64, cur.h, row0);
                    tma_store_3d(&tmap_out, src + 16384, 0, cur.h, row0 + 64);
                    tma_store_3d(&tmap_out, src + 24576, 64, cur.h, row0 + 64);
                    bulk_commit();
                }
            } else {
                char *const ob = reinterpret_cast<char *>(p.out);
                constexpr int kEsz = OUT == kOutF32 ? 4 : 2;
                constexpr int kRowsPerIt = OUT == kOutF32 ? 1 : 2;
                constexpr int kCols = OUT == kOutF32 ? 4 : 8;   // values per lane
                const int sub = lane / (32 / kRowsPerIt);
                const int cl = lane % (32 / kRowsPerIt);
                const int c0 = cl * kCols;                      // first column of this lane
#pragma unroll 4
                for (int it = 0; it < 32 / kRowsPerIt; ++it) {
                    const int rr = 32 * qd + kRowsPerIt * it + sub;
                    if (rr >= cur.L) continue;
                    const int rh = rr & 63;
                    float v[kCols];
                    const bool right = c0 >= 64;
                    const int cc = c0 & 63;
                    const float *src;
                    bool zero = false, mask = true;
                    if (rr < 64) {
                        src = M0 + rh * kC128Pitch + cc;
                        zero = right;
                    } else if (!right) {
                        src = M2 + rh * kC128Pitch + cc;
                        mask = false;
                    } else {
                        src = M1 + rh * kC128Pitch + cc;
                    }
#pragma unroll
                    for (int e4 = 0; e4 < kCols / 4; ++e4) {
                        const float4 x = *reinterpret_cast<const float4 *>(src + 4 * e4);
                        v[4 * e4 + 0] = x.x;
                        v[4 * e4 + 1] = x.y;
                        v[4 * e4 + 2] = x.z;
                        v[4 * e4 + 3] = x.w;
                    }
#pragma unroll
                    for (int e = 0; e < kCols; ++e)
                        if (zero || (mask && cc + e > rh)) v[e] = 0.0f;
                    char *dst = ob + ((cur.row0 + rr) * p.H + cur.h) * (128 * kEsz) + c0 * kEsz;
                    if (OUT == kOutF32) {
                        *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
                        uint4 u;
                        u.x = pack16x2<OUT>(v[0], v[1]);
                        u.y = pack16x2<OUT>(v[2], v[3]);
                        u.z = pack16x2<OUT>(v[4 % kCols], v[5 % kCols]);
                        u.w = pack16x2<OUT>(v[6 % kCols], v[7 % kCols]);
                        *reinterpret_cast<uint4 *>(dst) = u;
                    }
                }
            }
            cur = nx;
            rin = rnext;
        }
        if (kTmaOut && tid == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kC128Mma) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kC128TmemCols);
    }
}

// ------------------------------------------------------------ wait self-test
// One thread waits, through the kernels' bounded wait with a 20 ms limit, on a
// barrier phase that nothing completes; when the wait runs out it records
// GDR_ERR_TIMEOUT in the status word, as a pipeline wait of the kernels would.
constexpr uint64_t kProbeWaitNs = 20000000ull;

__global__ void bounded_wait_probe_kernel(int *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait_limited<kProbeWaitNs>(b, 0)) atomicExch(status, static_cast<int>(GDR_ERR_TIMEOUT));
    }
}

// ------------------------------------------------------ cu_seqlens contract
// Reads cu[0..B] and records GDR_ERR_CU_SEQLENS in the status word (unless an
// earlier status is still unread) when cu[0] != 0, some cu[n] > cu[n+1], or
// cu[B] > T.  Grid-stride over the B adjacent pairs; reads stay inside cu[0..B].
__global__ void check_cu_seqlens_kernel(const int32_t *cu, int64_t B, int64_t T, int *status) {
    bool bad = false;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; n < B; n += stride)
        bad |= __ldg(cu + n) > __ldg(cu + n + 1);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        bad |= __ldg(cu) != 0 || static_cast<int64_t>(__ldg(cu + B)) > T;
    if (bad) atomicCAS(status, static_cast<int>(GDR_OK), static_cast<int>(GDR_ERR_CU_SEQLENS));
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

using KernelFn = void (*)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap, Params);
using KernelFn128 = void (*)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap, Params);

template <int OUT, int MODE>
KernelFn kernel_for_nkb(int nkb) {
    switch (nkb) {
        case 1: return kkt_solve_kernel<OUT, 1, MODE>;
        case 2: return kkt_solve_kernel<OUT, 2, MODE>;
        case 3: return kkt_solve_kernel<OUT, 3, MODE>;
        default: return kkt_solve_kernel<OUT, 4, MODE>;
    }
}

KernelFn128 kernel_c128_for(int out_kind, int nkb) {
    if (out_kind == kOutBF16) return nkb == 1 ? kkt_solve_c128_kernel<kOutBF16, 1> : kkt_solve_c128_kernel<kOutBF16, 2>;
    if (out_kind == kOutF16) return nkb == 1 ? kkt_solve_c128_kernel<kOutF16, 1> : kkt_solve_c128_kernel<kOutF16, 2>;
    return nkb == 1 ? kkt_solve_c128_kernel<kOutF32, 1> : kkt_solve_c128_kernel<kOutF32, 2>;
}

// The instantiation for a mode, an output kind (gdr_dtype value) and K / 64.
KernelFn kernel_for(int mode, int out_kind, int nkb) {
    if (mode == kModeKkt) return kernel_for_nkb<kOutF32, kModeKkt>(nkb);
    if (mode == kModeSolve) {
        if (out_kind == kOutBF16) return kkt_solve_kernel<kOutBF16, 2, kModeSolve>;
        if (out_kind == kOutF16) return kkt_solve_kernel<kOutF16, 2, kModeSolve>;
        return kkt_solve_kernel<kOutF32, 2, kModeSolve>;
    }
    if (mode == kModeF32Keys) {   // nkb = K / 32: 2 or 4
        if (out_kind == kOutBF16) return nkb == 2 ? kkt_solve_kernel<kOutBF16, 2, kModeF32Keys> : kkt_solve_kernel<kOutBF16, 4, kModeF32Keys>;
        if (out_kind == kOutF16) return nkb == 2 ? kkt_solve_kernel<kOutF16, 2, kModeF32Keys> : kkt_solve_kernel<kOutF16, 4, kModeF32Keys>;
        return nkb == 2 ? kkt_solve_kernel<kOutF32, 2, kModeF32Keys> : kkt_solve_kernel<kOutF32, 4, kModeF32Keys>;
    }
    if (mode == kModeF32KeysTf32)   // bf16 output only; nkb = K / 32: 2 or 4
        return nkb == 2 ? kkt_solve_kernel<kOutBF16, 2, kModeF32KeysTf32> : kkt_solve_kernel<kOutBF16, 4, kModeF32KeysTf32>;
    if (out_kind == kOutBF16) return kernel_for_nkb<kOutBF16, kModeFused>(nkb);
    if (out_kind == kOutF16) return kernel_for_nkb<kOutF16, kModeFused>(nkb);
    return kernel_for_nkb<kOutF32, kModeFused>(nkb);
}

// Launch shape of the 64-token kernel in a mode: threads per CTA, dynamic
// shared memory and consumer warpgroups (the split fp32-key Gram has its own
// layout; every other mode shares one).
using SplitLayout = FusedLayout<kModeF32Keys>;
using BaseLayout = FusedLayout<kModeFused>;
static_assert(FusedLayout<kModeKkt>::kSmemBytes == BaseLayout::kSmemBytes &&
                  FusedLayout<kModeSolve>::kSmemBytes == BaseLayout::kSmemBytes &&
                  FusedLayout<kModeF32KeysTf32>::kSmemBytes == BaseLayout::kSmemBytes,
              "one layout for every mode but the split Gram");
int fused_threads(int mode) { return mode == kModeF32Keys ? SplitLayout::kThreads : BaseLayout::kThreads; }
int fused_smem(int mode) { return mode == kModeF32Keys ? SplitLayout::kSmemBytes : BaseLayout::kSmemBytes; }
int fused_wg(int mode) { return mode == kModeF32Keys ? SplitLayout::kNumWG : BaseLayout::kNumWG; }

constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_ready[kMaxDevices];   // 0 unknown, 1 ready, -1 unsupported
std::atomic<int> g_dev_sms[kMaxDevices];

// Scratch of the allocation-free chain entry point: room for A of at most
// kScratchTokenHeads token-heads (64 fp32 values each, 64 MiB in total).  It is
// part of the library's device image, so every GPU that loads the library
// holds it until the process exits.
constexpr int64_t kScratchTokenHeads = int64_t(1) << 18;
static __device__ __align__(256) float g_chain_scratch[kScratchTokenHeads * 64];

// Device address of g_chain_scratch, looked up once per device with that device
// current.  In host code the array's name stands for a host-side shadow, not
// for device memory, so the address must come from cudaGetSymbolAddress.
std::atomic<float *> g_scratch_addr[kMaxDevices];

int scratch_for_current_device(float **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GDR_ERR_DEVICE;
    }
    float *a = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        void *sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_chain_scratch) != cudaSuccess || sym == nullptr) {
            cudaGetLastError();
            return GDR_ERR_CUDA;
        }
        a = static_cast<float *>(sym);
        g_scratch_addr[dev].store(a, std::memory_order_release);
    }
    *addr = a;
    return GDR_OK;
}

int prepare_device(int *sms) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GDR_ERR_DEVICE;
    }
    int st = g_dev_ready[dev].load(std::memory_order_acquire);
    if (st == 0) {
        int major = 0, minor = 0, nsm = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GDR_ERR_DEVICE;
        }
        if (major != 10 || minor != 3) {
            g_dev_ready[dev].store(-1, std::memory_order_release);
            return GDR_ERR_DEVICE;
        }
        bool attr_ok = true;
        for (int m = 0; m < 3; ++m)
            for (int o = 0; o < 3; ++o)
                for (int n = 1; n <= 4; ++n)
                    attr_ok = attr_ok && cudaFuncSetAttribute(kernel_for(m, o, n),
                                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                              fused_smem(m)) == cudaSuccess;
        for (int o = 0; o < 3; ++o)
            for (int n = 2; n <= 4; n += 2)
                attr_ok = attr_ok && cudaFuncSetAttribute(kernel_for(kModeF32Keys, o, n),
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          fused_smem(kModeF32Keys)) == cudaSuccess;
        for (int n = 2; n <= 4; n += 2)
            attr_ok = attr_ok && cudaFuncSetAttribute(kernel_for(kModeF32KeysTf32, kOutBF16, n),
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                      fused_smem(kModeF32KeysTf32)) == cudaSuccess;
        for (int o = 0; o < 3; ++o)
            for (int n = 1; n <= 2; ++n)
                attr_ok = attr_ok && cudaFuncSetAttribute(kernel_c128_for(o, n),
                                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                          kC128SmemBytes) == cudaSuccess;
        if (!attr_ok) {
            cudaGetLastError();
            return GDR_ERR_CUDA;
        }
        g_dev_sms[dev].store(nsm, std::memory_order_relaxed);
        g_dev_ready[dev].store(1, std::memory_order_release);
        st = 1;
    }
    if (st < 0) return GDR_ERR_DEVICE;
    *sms = g_dev_sms[dev].load(std::memory_order_relaxed);
    return GDR_OK;
}

}  // namespace gdr

extern "C" {

const char *gdr_status_string(int status) {
    switch (status) {
        case GDR_OK: return "ok";
        case GDR_ERR_NULL: return "a required pointer is NULL";
        case GDR_ERR_SHAPE:
            return "unsupported or inconsistent sizes (K in {64, 128, 192, 256}; K <= 128 for fp32 keys and for "
                   "chunk 128; B*T < 2^31)";
        case GDR_ERR_CHUNK: return "chunk_size must be 64 (or 128 for the fused call, K <= 128)";
        case GDR_ERR_DTYPE:
            return "unsupported dtype (k: bf16 or fp16, or fp32 with K in {64, 128} in the fused chunk-64 call; "
                   "beta: fp32, bf16 or fp16; out: fp32, bf16 or fp16)";
        case GDR_ERR_ALIGN: return "pointer misaligned (k and out 16 B, g 4 B, beta 2 B, cu_seqlens 4 B)";
        case GDR_ERR_DEVICE: return "no usable CUDA device (an sm_103 GPU is required)";
        case GDR_ERR_CUDA: return "a CUDA runtime or driver call failed";
        case GDR_ERR_TIMEOUT: return "a device-side pipeline wait timed out";
        case GDR_ERR_SCRATCH:
            return "problem too large for the allocation-free entry point (at most 262144 token-heads)";
        case GDR_ERR_CU_SEQLENS:
            return "cu_seqlens breaks its contract (cu[0] = 0, non-decreasing, cu[B] <= T)";
        default: return "unknown gdr_status";
    }
}

}  // extern "C"

namespace gdr {

// Validates the arguments and enqueues one launch of the given mode.  `in` is
// the key tensor (fused and kkt modes; in_dtype bf16 or fp16, K columns) or the
// fp32 A tensor (solve mode; 64 columns).  The kkt mode writes fp32 A to `out`.
// Host-side argument checks of one launch; GDR_OK means a launch may follow
// (or, for an empty problem, that nothing needs to run: see is_empty).
int validate(int mode, const void *in, int in_dtype, const void *g, const void *beta, int beta_dtype,
             const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H, int64_t K, int chunk_size,
             int out_dtype, const void *out) {
    // Chunk 128: the fused call only, K = 64 or 128.
    if (chunk_size != kChunk && !(chunk_size == 128 && mode == kModeFused)) return GDR_ERR_CHUNK;
    if (chunk_size == 128 && K > 128) return GDR_ERR_SHAPE;
    // Keys: bf16 or fp16; fp32 keys for the fused chunk-64 call only (K = 64 or 128).
    const bool f32_keys = mode == kModeFused && in_dtype == GDR_F32;
    if (mode == kModeSolve ? in_dtype != GDR_F32
                           : (in_dtype != GDR_BF16 && in_dtype != GDR_F16 && !f32_keys))
        return GDR_ERR_DTYPE;
    if (f32_keys && chunk_size != kChunk) return GDR_ERR_DTYPE;
    if (f32_keys && K > 128) return GDR_ERR_SHAPE;
    if (beta && beta_dtype != GDR_F32 && beta_dtype != GDR_BF16 && beta_dtype != GDR_F16)
        return GDR_ERR_DTYPE;
    if (out_dtype != GDR_F32 && out_dtype != GDR_BF16 && out_dtype != GDR_F16) return GDR_ERR_DTYPE;
    if (B < 0 || T < 0 || H < 0 || K < 64 || K > kMaxHeadK || K % 64 != 0) return GDR_ERR_SHAPE;
    if (B == 0 || T == 0 || H == 0) return GDR_OK;
    if (!in || !out) return GDR_ERR_NULL;
    const int64_t ntok = cu_seqlens ? T : B * T;
    if (B > (int64_t(1) << 31) || T > (int64_t(1) << 31) || ntok >= (int64_t(1) << 31) ||
        H > (int64_t(1) << 24) || (cu_seqlens == nullptr && B > ((int64_t(1) << 31) / T)))
        return GDR_ERR_SHAPE;
    const uintptr_t beta_align = (beta && beta_dtype == GDR_F32) ? 3 : 1;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) ||
        (reinterpret_cast<uintptr_t>(g) & 3) || (reinterpret_cast<uintptr_t>(beta) & beta_align) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens) & 3))
        return GDR_ERR_ALIGN;
    return GDR_OK;
}

bool is_empty(int64_t B, int64_t T, int64_t H) { return B == 0 || T == 0 || H == 0; }

int launch(int mode, const void *in, int in_dtype, const float *g, const void *beta, int beta_dtype,
           const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H, int64_t K, int chunk_size,
           int out_dtype, void *out, void *stream) {
    int rc = validate(mode, in, in_dtype, g, beta, beta_dtype, cu_seqlens, B, T, H, K, chunk_size,
                      out_dtype, out);
    if (rc != GDR_OK || is_empty(B, T, H)) return rc;
    const int64_t ntok = cu_seqlens ? T : B * T;

    int sms = 0;
    rc = prepare_device(&sms);
    if (rc != GDR_OK) return rc;
    auto encode = encode_fn();
    if (!encode) return GDR_ERR_CUDA;

    // fp32 keys run their own kernel mode.
    const int kmode = (mode == kModeFused && in_dtype == GDR_F32)
                          ? (out_dtype == GDR_BF16 ? kModeF32KeysTf32 : kModeF32Keys)
                          : mode;
    // Input tiles: 64 rows x 128 bytes per box (64 bf16/fp16 key columns, or 32
    // fp32 columns of keys or of A), 128-byte swizzle.
    CUtensorMap tmap;
    {
        const int esz = in_dtype == GDR_F32 ? 4 : 2;
        const int64_t cols = mode == kModeSolve ? 64 : K;
        const CUtensorMapDataType dt = in_dtype == GDR_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : in_dtype == GDR_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(H),
                                    static_cast<cuuint64_t>(ntok)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * esz),
                                       static_cast<cuuint64_t>(H * cols * esz)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), 1, static_cast<cuuint32_t>(kChunk)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmap, dt, 3, const_cast<void *>(in), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GDR_ERR_CUDA;
    }
    const int out_kind = mode == kModeKkt ? GDR_F32 : out_dtype;
    CUtensorMap tmap_o = {};
    if (chunk_size == kChunk) {
        const int esz = out_kind == GDR_F32 ? 4 : 2;
        const CUtensorMapDataType odt = out_kind == GDR_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                        : out_kind == GDR_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const cuuint64_t odims[3] = {64, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(ntok)};
        const cuuint64_t ostr[2] = {static_cast<cuuint64_t>(64 * esz), static_cast<cuuint64_t>(H * 64 * esz)};
        const cuuint32_t obox[3] = {static_cast<cuuint32_t>(128 / esz), 1, static_cast<cuuint32_t>(kChunk)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmap_o, odt, 3, out, odims, ostr, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GDR_ERR_CUDA;
    } else if (out_kind != GDR_F32) {
        // Chunk 128, 16-bit output: rows of 128 values, 64 x 64 boxes of 128-byte rows.
        const CUtensorMapDataType odt = out_kind == GDR_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const cuuint64_t odims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(ntok)};
        const cuuint64_t ostr[2] = {static_cast<cuuint64_t>(128 * 2), static_cast<cuuint64_t>(H * 128 * 2)};
        const cuuint32_t obox[3] = {64, 1, static_cast<cuuint32_t>(kChunk)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tmap_o, odt, 3, out, odims, ostr, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return GDR_ERR_CUDA;
    }

    Params prm;
    prm.g = mode == kModeSolve ? nullptr : g;
    prm.beta = mode == kModeSolve ? nullptr : beta;
    prm.beta_kind = prm.beta ? beta_dtype : GDR_F32;
    prm.idesc = in_dtype == GDR_F32 ? kIdescTf32 : idesc_f16_kind(in_dtype == GDR_BF16);
    prm.cu = cu_seqlens;
    prm.out = out;
    prm.B = B;
    prm.T = T;
    prm.H = H;
    const int64_t CH = chunk_size;                 // 64, or 128 (one chunk per pipeline pair)
    prm.NT = (T + CH - 1) / CH;
    prm.n_slots = cu_seqlens ? (T + (CH - 1) * B) / CH : B * prm.NT;
    if (prm.n_slots * H >= (int64_t(1) << 31)) return GDR_ERR_SHAPE;
    prm.n_pairs = CH == 128 ? prm.n_slots * H : (prm.n_slots * H + 1) / 2;
    prm.divH = make_fastdiv(static_cast<uint32_t>(H));
    prm.divNT = make_fastdiv(static_cast<uint32_t>(prm.NT));
    int *status_ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status_ptr), g_status_word) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    prm.status = status_ptr;

    const int64_t grid = prm.n_pairs < sms ? prm.n_pairs : sms;
    // Tile strides of a CTA's and of a warpgroup's consecutive pairs.
    const int64_t per_pair = CH == 128 ? 1 : 2;
    const int64_t n_wg = CH == 128 ? kC128WG : fused_wg(kmode);
    prm.pair_ds = static_cast<uint32_t>((per_pair * grid) / H);
    prm.pair_dh = static_cast<uint32_t>((per_pair * grid) % H);
    prm.wg_ds = static_cast<uint32_t>((per_pair * grid * n_wg) / H);
    prm.wg_dh = static_cast<uint32_t>((per_pair * grid * n_wg) % H);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Programmatic stream serialization: the kernel may be scheduled while the
    // stream's previous grid drains; it waits (griddepcontrol.wait) for that
    // grid before touching global memory, so only its set-up overlaps.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (CH == 128) {
        cfg.blockDim = dim3(kC128Threads);
        cfg.dynamicSmemBytes = kC128SmemBytes;
        err = cudaLaunchKernelEx(&cfg, kernel_c128_for(out_kind, static_cast<int>(K / 64)), tmap, tmap_o, prm);
    } else {
        const int nkb = static_cast<int>(in_dtype == GDR_F32 && kmode != kModeSolve ? K / 32 : K / 64);
        cfg.blockDim = dim3(fused_threads(kmode));
        cfg.dynamicSmemBytes = fused_smem(kmode);
        err = cudaLaunchKernelEx(&cfg, kernel_for(kmode, out_kind, nkb), tmap, tmap_o, prm);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    return GDR_OK;
}

}  // namespace gdr

extern "C" {

int gdr_kkt_solve_ex(const void *k, int k_dtype, const float *g, const void *beta, int beta_dtype,
                     const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H, int64_t K,
                     int chunk_size, int out_dtype, void *out, void *stream) {
    return gdr::launch(gdr::kModeFused, k, k_dtype, g, beta, beta_dtype, cu_seqlens, B, T, H, K,
                       chunk_size, out_dtype, out, stream);
}

int gdr_chunk_scaled_dot_kkt(const void *k, int k_dtype, const float *g, const void *beta,
                             int beta_dtype, const int32_t *cu_seqlens, int64_t B, int64_t T,
                             int64_t H, int64_t K, int chunk_size, float *A, void *stream) {
    return gdr::launch(gdr::kModeKkt, k, k_dtype, g, beta, beta_dtype, cu_seqlens, B, T, H, K,
                       chunk_size, GDR_F32, A, stream);
}

int gdr_solve_tril(const float *A, const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                   int chunk_size, int out_dtype, void *out, void *stream) {
    return gdr::launch(gdr::kModeSolve, A, GDR_F32, nullptr, nullptr, GDR_F32, cu_seqlens, B, T, H,
                       64, chunk_size, out_dtype, out, stream);
}

int gdr_kkt_solve_unfused_noalloc(const void *k, int k_dtype, const float *g, const void *beta,
                                  int beta_dtype, const int32_t *cu_seqlens, int64_t B, int64_t T,
                                  int64_t H, int64_t K, int chunk_size, int out_dtype, void *out,
                                  void *stream) {
    using namespace gdr;
    // The argument checks of both halves (with a stand-in, aligned scratch
    // address), then the size limit; nothing is allocated anywhere on this path.
    const float *const stand_in = reinterpret_cast<const float *>(uintptr_t(256));
    int rc = validate(kModeKkt, k, k_dtype, g, beta, beta_dtype, cu_seqlens, B, T, H, K, chunk_size,
                      GDR_F32, stand_in);
    if (rc == GDR_OK)
        rc = validate(kModeSolve, stand_in, GDR_F32, nullptr, nullptr, GDR_F32, cu_seqlens, B, T, H, 64,
                      chunk_size, out_dtype, out);
    if (rc != GDR_OK || is_empty(B, T, H)) return rc;
    const int64_t ntok = cu_seqlens ? T : B * T;
    if (ntok > kScratchTokenHeads || H > kScratchTokenHeads / ntok) return GDR_ERR_SCRATCH;
    float *A = nullptr;
    rc = scratch_for_current_device(&A);
    if (rc != GDR_OK) return rc;
    rc = gdr_chunk_scaled_dot_kkt(k, k_dtype, g, beta, beta_dtype, cu_seqlens, B, T, H, K, chunk_size,
                                  A, stream);
    if (rc != GDR_OK) return rc;
    return gdr_solve_tril(A, cu_seqlens, B, T, H, chunk_size, out_dtype, out, stream);
}

int gdr_kkt_solve(const void *k, const float *g, const void *beta, const int32_t *cu_seqlens,
                  int64_t B, int64_t T, int64_t H, int64_t K, int chunk_size, int out_dtype,
                  void *out, void *stream) {
    return gdr_kkt_solve_ex(k, GDR_BF16, g, beta, GDR_BF16, cu_seqlens, B, T, H, K, chunk_size,
                            out_dtype, out, stream);
}

int gdr_kkt_solve_device_status(int *status) {
    if (!status) return GDR_ERR_NULL;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, gdr::g_status_word, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    const int zero = 0;
    if (cudaMemcpyToSymbol(gdr::g_status_word, &zero, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    *status = v;
    return GDR_OK;
}

int gdr_selftest_bounded_wait(void *stream) {
    using namespace gdr;
    int sms = 0;
    int rc = prepare_device(&sms);
    if (rc != GDR_OK) return rc;
    int *status_ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status_ptr), g_status_word) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status_ptr);
    if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
    return GDR_OK;
}

int gdr_check_cu_seqlens(const int32_t *cu_seqlens, int64_t B, int64_t T, void *stream) {
    using namespace gdr;
    if (!cu_seqlens) return GDR_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3) return GDR_ERR_ALIGN;
    if (B < 0 || T < 0 || B >= (int64_t(1) << 31)) return GDR_ERR_SHAPE;
    int sms = 0;
    int rc = prepare_device(&sms);
    if (rc != GDR_OK) return rc;
    int *status_ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status_ptr), g_status_word) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    const int64_t blocks = (B + 255) / 256;
    const int64_t cap = 4 * static_cast<int64_t>(sms);
    const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
    check_cu_seqlens_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(cu_seqlens, B, T, status_ptr);
    if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
    return GDR_OK;
}

int gdr_kkt_solve_num_sms(void) {
    int sms = 0;
    int rc = gdr::prepare_device(&sms);
    return rc == GDR_OK ? sms : rc;
}

}  // extern "C"
