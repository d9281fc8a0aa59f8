// INT8 x INT8 -> INT32 GEMM with fused dequant on a pair of SMs, the weight
// codes widened on chip into tensor memory (no weight image in HBM).
//
// What it computes (Cider README, "Metal Kernel Pipeline" and
// "Quantization"; W4A8 per the "Modes" table, "Unpack -> TensorOps"):
// acc[m,n] = sum_k q[m,k] * wq[n,k] exactly in int32, then
//   per-channel: y = fp16(((float)acc * s_a[m]) * s_w[n])
//   per-group:   f = sum over groups g, ascending, of (float)P_g * s_w[n,g]; y = fp16(f * s_a[m])
// on exact fp16 images of the codes with tcgen05 kind::f16 (sm_103a has no
// integer MMA kind) and an fp32 tensor-memory accumulator folded into int32
// every <= 1024 k (every group in per-group mode), where every partial sum is
// an exact integer.
//
// Roles are swapped relative to a token-major GEMM: the weights are the MMA's
// A operand (M = 256 output channels per SM pair, 128 per CTA) and the tokens
// its B operand (N = 192 tokens per pair tile for many tokens, 96 loaded by
// each CTA; 128 for at most 128 tokens). The
// tensor core reads A from tensor memory, so the weights never need an fp16
// copy in shared or global memory: TMA stages each CTA's raw codes (INT8
// [N,K], or packed INT4 [N,K/2]) as 128 rows x one 64-k block, and four
// converter warps (one per TMEM lane quadrant; thread = weight row) widen
// them to exact fp16 pairs with byte permutes and one fp16 subtraction and
// write them with tcgen05.st into one of four 32-column A stages in TMEM. The
// activations come from the fp16 code image of the per-token quantization
// (K-major, 128-byte swizzle) as B. The even CTA's MMA thread issues
// tcgen05.mma.cta_group::2 (M 256, N 192, K 16) with A in both CTAs' tensor
// memory and B in both CTAs' shared memory, into two 192-column fp32
// accumulators per CTA (lane = output channel, column = token). Measured on
// B300: this MMA runs at full rate (96 cycles per instruction), the same as
// with A in shared memory, but each tcgen05.mma costs the issuing thread
// about 55 cycles and each tcgen05.commit about 60, so a k-block (four MMAs,
// 384 cycles) carries exactly one barrier wait and one commit: the token
// bytes and the converters' arrivals complete one "full" barrier, and one
// commit per k-block frees both its shared-memory stage and its A stage.
//
// Epilogue (8 warps: each one TMEM lane quadrant, i.e. 32 output channels,
// and half of the tile's 192 tokens): segment folds as in the token-major
// kernels; the final dequant writes 32 tokens x 32 channels per step through
// shared-memory staging and a TMA store. Persistent over tiles (the faster
// tile index chosen so that concurrent clusters share the larger operand in
// L2). Few tokens: per-channel layers may instead cut the k-blocks of all
// tiles into one equal run per pair (stream-K); a tile shared by pairs is
// stored by each CTA as an int32 partial and summed by
// sk_fixup_pair_kernel. Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {
namespace gemmw {

constexpr int BW = 128;           // weight rows per CTA (MMA M = 256 per pair)
constexpr int BT_MANY = 192;      // tokens per pair tile (MMA N) for many tokens
constexpr int BT_FEW = 128;       // ... and for at most 128 tokens; each CTA loads BT / 2
constexpr int BK = 64;            // k per block: one 128-byte swizzle row of fp16 tokens
constexpr int KB_PER_STAGE = 1;   // 64-k blocks per stage (the MMA loop assumes 1)
constexpr int SK = BK * KB_PER_STAGE;
constexpr int STAGES = 8 / KB_PER_STAGE;    // shared-memory ring (raw weights + tokens)
constexpr int A_STAGES = 4 / KB_PER_STAGE;  // tensor-memory ring of widened weights
constexpr int A_STAGE_COLS = SK / 2;  // two fp16 per 32-bit column
constexpr int NUM_ACC = 2;
constexpr int TMEM_COLS = 512;
constexpr int RAW_STAGE_BYTES = BW * SK;            // 16 KB (INT8; INT4 uses half)
constexpr int MAX_SEG_KB = 16;    // 16 x 64 = 1024 k per exact fp32 segment
// Warps 0-3: TMA producer, MMA issuer (and TMEM owner), two idle; warps
// 4-11: two converter warpgroups, taking alternate k-blocks; warps 12-19:
// epilogue.
constexpr int NUM_CONV_GROUPS = 2;
constexpr int FIRST_EPI_WARP = 4 + 4 * NUM_CONV_GROUPS;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = (FIRST_EPI_WARP + NUM_EPI_WARPS) * 32;
constexpr int LAUNCH_REGS = 96;
constexpr int ROLE_REGS = 40;
// Converter / epilogue register split per weight width (the split ptxas
// allocates without spills for the per-channel kernels of each width).
template <int BITS>
struct Regs {
    static constexpr int kConv = BITS == 8 ? 56 : 48;
    static constexpr int kEpi = BITS == 8 ? 160 : 168;
    static_assert(128 * ROLE_REGS + 128 * NUM_CONV_GROUPS * kConv + 256 * kEpi <=
                      NUM_THREADS * LAUNCH_REGS,
                  "register split exceeds the launch allocation");
};
constexpr int LD = 16;            // columns per TMEM load of the fold
constexpr int OUT_WARP_BYTES = 32 * 64;  // staging: 32 tokens x 32 channels fp16
constexpr int SMEM_LIMIT = 232448;
constexpr uint16_t kPairMask = 0x3;

struct __align__(8) Barriers {
    // even CTA: stage u's token blocks landed (both CTAs' TMA bytes) and its
    // weights are in A stage u % A_STAGES (both CTAs' converters arrived):
    // one producer arrival with the byte count + 4 converter warps x 2 CTAs.
    uint64_t full[STAGES];
    // each CTA: the MMAs of stage u completed (one commit, multicast): the
    // shared-memory stage, and A stage u % A_STAGES, may be refilled.
    uint64_t empty[STAGES];
    uint64_t raw_full[STAGES];   // each CTA: its raw weight block landed
    uint64_t acc_full[NUM_ACC];  // each CTA: accumulator buffer ready
    uint64_t acc_empty[NUM_ACC]; // even CTA: both CTAs' epilogues drained it (16 warps)
    uint64_t drain;              // even CTA: MMA drain after an abort
};
static_assert(sizeof(Barriers) <= 512, "barrier area");
static_assert(STAGES % A_STAGES == 0 && STAGES >= A_STAGES, "A stages follow the ring");

// Shapes that depend on the token tile BT.
template <int BT>
struct Tile {
    static constexpr int ACC_COLS = BT;
    static constexpr int A_COL0 = NUM_ACC * ACC_COLS;  // 384 for BT 192
    static_assert(A_COL0 + A_STAGES * A_STAGE_COLS <= TMEM_COLS, "tensor memory budget");
    static constexpr int ACT_BLOCK_BYTES = (BT / 2) * BK * 2;  // one 64-k token block per CTA
    static constexpr int ACT_STAGE_BYTES = KB_PER_STAGE * ACT_BLOCK_BYTES;
    static constexpr int COLS = BT / 2;       // tokens per epilogue warp
    static constexpr int CHUNKS = COLS / 32;  // 32-token output rounds per warp
    static_assert(COLS % 32 == 0 && COLS % LD == 0, "epilogue rounds");
};
static_assert(SK == 64 || SK == 128, "raw rows of 32 to 128 bytes");
static_assert(KB_PER_STAGE == 1 && (STAGES & (STAGES - 1)) == 0 &&
                  (A_STAGES & (A_STAGES - 1)) == 0 && (NUM_ACC & (NUM_ACC - 1)) == 0,
              "ring arithmetic by masks");

template <int BT>
struct SmemLayout {
    static constexpr int ACT_STAGE_BYTES = Tile<BT>::ACT_STAGE_BYTES;
    static constexpr int raw_off = 0;
    static constexpr int act_off = raw_off + STAGES * RAW_STAGE_BYTES;
    static constexpr int out_off = act_off + STAGES * ACT_STAGE_BYTES;
    static constexpr int bar_off = out_off + NUM_EPI_WARPS * OUT_WARP_BYTES;
    static constexpr int misc_off = bar_off + 512;  // tmem base, abort flag
    static constexpr int bytes = misc_off + 16;
    static constexpr int alloc_bytes = bytes + 1024;  // runtime 1024-byte alignment slack
    static_assert(alloc_bytes <= SMEM_LIMIT, "shared memory per block");
    static_assert(act_off % 1024 == 0 && RAW_STAGE_BYTES % 1024 == 0 &&
                      ACT_STAGE_BYTES % 1024 == 0,
                  "swizzled stages must stay 1024-byte aligned");
};

struct Params {
    int M, N, K;
    int bits;        // 8: INT8 codes; 4: packed INT4 (nibble = code + 8)
    int num_kb;
    int seg_kb;      // k-blocks per segment (one accumulator buffer)
    int num_seg;
    int G;
    int tiles_t, tiles_w;  // token tiles of BT, weight tiles of 2 * BW
    int w_fastest;         // tile order (tile_coords)
    // Stream-K (per-channel, one token tile): the tiles' k-blocks in tile
    // order form `units` units; pair c takes [c * units / pairs, (c + 1) *
    // units / pairs). A tile several pairs share is stored by each CTA as an
    // int32 partial [part_rows tokens][BW channels] in `part` (slot 0: the
    // pair's first item, 1: its last) and summed by sk_fixup_pair_kernel.
    int streamk;
    int64_t units;
    int32_t* part;
    int part_rows;
    const float* s_a;
    const float* s_w;
    void* out;
    int tma_store;   // 16-bit output through tmap_y (N % 8 == 0)
    int out_bf16;
    uint64_t timeout_ns;
    unsigned long long* status;
};

enum : uint32_t {
    kSiteProducerEmpty = 0x401,
    kSiteMmaAccEmpty = 0x403,
    kSiteMmaFull = 0x404,
    kSiteConvRaw = 0x406,
    kSiteConvA = 0x407,
    kSiteEpiAccFull = 0x408,
    kSiteDrain = 0x409,
    kSiteProducerDrain = 0x40a,
};

// A pair's work item: k-blocks [kb0, kb1) of one tile.
struct Work {
    int tile, kb0, kb1;
};

// The items of this pair, in order: whole tiles cluster, + nclusters, ...;
// or with stream-K (kernels built with SK) its run of units, cut at tile
// boundaries.
template <bool SK>
struct WorkIter {
    int64_t u, uend;
    int tile, num_tiles, step, nk;
    bool sk;
    __device__ __forceinline__ WorkIter(const Params& p, int cluster, int nclusters, int num_tiles_)
        : tile(cluster), num_tiles(num_tiles_), step(nclusters), nk(p.num_kb),
          sk(SK && p.streamk != 0) {
        u = sk ? (int64_t)cluster * p.units / nclusters : 0;
        uend = sk ? ((int64_t)cluster + 1) * p.units / nclusters : 0;
    }
    __device__ __forceinline__ bool next(Work& w) {
        if (SK && sk) {
            if (u >= uend) return false;
            w.tile = (int)(u / nk);
            w.kb0 = (int)(u - (int64_t)w.tile * nk);
            const int64_t left = uend - u;
            w.kb1 = (left < (int64_t)(nk - w.kb0)) ? w.kb0 + (int)left : nk;
            u += w.kb1 - w.kb0;
            return true;
        }
        if (tile >= num_tiles) return false;
        w.tile = tile;
        w.kb0 = 0;
        w.kb1 = nk;
        tile += step;
        return true;
    }
};

// Segments of an item: per-group, one group each (items are whole tiles);
// per-channel, the item's k-blocks in equal runs of at most MAX_SEG_KB.
template <GemmMode MODE, int MAX_SEG>
__device__ __forceinline__ void item_segments(const Params& p, const Work& w, int& seg_kb,
                                              int& nseg) {
    if constexpr (MODE == GemmMode::kPgF16 || MODE == GemmMode::kRawPgS32) {
        seg_kb = p.seg_kb;
        nseg = p.num_seg;
    } else {
        const int len = w.kb1 - w.kb0;
        const int n = (len + MAX_SEG - 1) / MAX_SEG;
        seg_kb = (len + n - 1) / n;
        nseg = (len + seg_kb - 1) / seg_kb;
    }
}

// Tile order: weight tiles fastest when the activation image is the larger
// operand (concurrent clusters then share token tiles, and the activations
// are read from DRAM about once), token tiles fastest otherwise.
__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& tt, int& tw) {
    if (p.w_fastest) {
        tw = tile % p.tiles_w;
        tt = tile / p.tiles_w;
    } else {
        tt = tile % p.tiles_t;
        tw = tile / p.tiles_t;
    }
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T on both CTAs of the pair, kind::f16.
__device__ __forceinline__ void mma_pair_a_tmem(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The four MMAs of one 64-k block: D (+)= A[a_tmem + 8k] * B[b_desc + 2k]^T
// for k = 0..3 (16 k each; B advances 32 bytes within its 128-byte swizzle
// rows), the first one accumulating only if `accumulate`.
__device__ __forceinline__ void mma4_pair_a_tmem(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %4, %4;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%5], %6, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%7], %8, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%9], %10, %3, t;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(a_tmem + 8), "l"(b_desc + 2),
        "r"(a_tmem + 16), "l"(b_desc + 4), "r"(a_tmem + 24), "l"(b_desc + 6)
        : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes from 32 registers.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 16 consecutive TMEM columns of this warp's 32 lanes from 16 registers.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Four signed INT8 codes (k order) -> two packed fp16 pairs (exact): the code
// plus 128 goes under the fp16 exponent of 1024 (0x64 high byte), then
// 1024 + 128 is subtracted.
__device__ __forceinline__ void widen_i8x4(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // [c0 + 128, 0x64, c1 + 128, 0x64]
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // [c2 + 128, 0x64, c3 + 128, 0x64]
    const __half2 bias = __float2half2_rn(1152.0f);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    p01 = *reinterpret_cast<const uint32_t*>(&ha);
    p23 = *reinterpret_cast<const uint32_t*>(&hb);
}

// Eight INT4 codes (one 32-bit word: element 2j in the low nibble of byte j)
// -> four packed fp16 pairs (exact): nibble under the exponent of 1024, then
// 1024 + 8 subtracted.
__device__ __forceinline__ void widen_i4x8(uint32_t w, uint32_t* p) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // elements 0, 2, 4, 6
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // elements 1, 3, 5, 7
    const __half2 bias = __float2half2_rn(1032.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // bytes [lo.bj, hi.bj] -> halves 0x64lo, 0x64hi
        const uint32_t sel = (uint32_t)j | ((uint32_t)(4 + j) << 8);
        uint32_t v = (__byte_perm(lo, hi, sel) & 0x00FF00FFu) | 0x64006400u;
        const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v), bias);
        p[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
}

template <GemmMode MODE, int BITS, int BT, int KPS_, int GPS>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(LAUNCH_REGS)
    gemm_tw_kernel(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_y, const Params p) {
    using SmemLayout = gemmw::SmemLayout<BT>;
    constexpr int ACC_COLS = Tile<BT>::ACC_COLS;
    constexpr int A_COL0 = Tile<BT>::A_COL0;
    constexpr int ACT_BLOCK_BYTES = Tile<BT>::ACT_BLOCK_BYTES;
    constexpr int ACT_STAGE_BYTES_1 = Tile<BT>::ACT_STAGE_BYTES;  // one 64-k block
    constexpr int COLS = Tile<BT>::COLS;
    constexpr int CHUNKS = Tile<BT>::CHUNKS;
    // Stream-K is built into the few-token per-channel kernels only.
    constexpr bool kStreamK =
        (BT == BT_FEW) && (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32);
    using WorkIter = gemmw::WorkIter<kStreamK>;
    // KPS 64-k blocks per stage: two for the few-token per-channel kernels
    // and for per-group layers whose groups are whole stages (a multiple of
    // 128 k), one otherwise. With two, the MMA thread waits and commits once
    // per eight MMAs (tcgen05.mma holds its issuing thread until the tensor
    // core takes it, so every wait, commit and loop step of that thread adds
    // to the time of a k-block), and the "k-blocks" of Params (num_kb,
    // segments, stream-K units) count stages of 128 k.
    constexpr int KPS = KPS_;
    static_assert(KPS == 1 || KPS == 2, "one or two k-blocks per stage");
    // GPS = 2: per-group layers of one k-block per group with two k-blocks
    // per stage, i.e. two groups per stage, each into its own accumulator
    // buffer; Params count stages in num_kb and groups in num_seg.
    static_assert(GPS == 1 || (GPS == 2 && KPS == 2 &&
                               (MODE == GemmMode::kPgF16 || MODE == GemmMode::kRawPgS32)),
                  "two groups per stage: per-group kernels with two k-blocks per stage");
    static_assert(!kStreamK || KPS == 2, "the stream-K kernels take two k-blocks per stage");
    constexpr int SK = BK * KPS;                  // k per stage
    constexpr int STAGES = 8 / KPS;               // the same shared-memory bytes
    constexpr int A_STAGES = 4 / KPS;             // the same tensor-memory columns
    constexpr int A_STAGE_COLS = SK / 2;
    constexpr int RAW_STAGE_BYTES = BW * SK;
    constexpr int MAX_SEG = MAX_SEG_KB / KPS;
    constexpr int ACT_STAGE_BYTES = KPS * ACT_STAGE_BYTES_1;
    constexpr int RAW_ROW = (BITS == 8) ? SK : SK / 2;  // raw bytes of one row and stage
    constexpr int RAW_BYTES = BW * RAW_ROW;
    static_assert(ACT_STAGE_BYTES == KPS * ACT_BLOCK_BYTES, "token blocks per stage");
    static_assert(STAGES * RAW_STAGE_BYTES == gemmw::STAGES * gemmw::RAW_STAGE_BYTES &&
                      STAGES * ACT_STAGE_BYTES == gemmw::STAGES * ACT_STAGE_BYTES_1 &&
                      A_STAGES * A_STAGE_COLS == gemmw::A_STAGES * gemmw::A_STAGE_COLS,
                  "the stage rings keep their byte and column budgets");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bars = reinterpret_cast<Barriers*>(smem + SmemLayout::bar_off);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + SmemLayout::misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::misc_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int cluster = (int)cluster_id_x();
    const int nclusters = (int)num_clusters_x();
    const int num_tiles = p.tiles_t * p.tiles_w;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1 + 4 * 2);
            mbar_init(smem_u32(&bars->empty[s]), 1);
            mbar_init(smem_u32(&bars->raw_full[s]), 1);
        }
        for (int b = 0; b < NUM_ACC; ++b) {
            mbar_init(smem_u32(&bars->acc_full[b]), 1);
            mbar_init(smem_u32(&bars->acc_empty[b]), 2 * NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_x);
        prefetch_tmap(&tmap_w);
        if (p.tma_store) prefetch_tmap(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_base_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // Both CTAs' barriers are initialised before any cross-CTA arrive or TMA.
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_slot;
    // Everything above overlaps the tail of the preceding kernel (programmatic
    // dependent launch); global memory is touched only after this wait.
    grid_dep_wait();
    grid_dep_launch();

    if (warp < 4) {
        setmaxnreg_dec<ROLE_REGS>();
        if (warp == 0 && lane == 0) {
            // ------------------------------ TMA producer (both CTAs) ----------
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            WorkIter it(p, cluster, nclusters, num_tiles);
            Work wk;
            while (it.next(wk)) {
                int tt, tw;
                tile_coords(p, wk.tile, tt, tw);
                const int w_row = tw * (2 * BW) + (int)rank * BW;
                const int t_row = tt * BT + (int)rank * (BT / 2);
                for (int ks = wk.kb0; ks < wk.kb1; ++ks) {
                    // The MMAs of the stage's previous use completed: its token
                    // blocks were read, and so was its raw block (the
                    // converters arrive on the full barrier the MMA waited on).
                    if (!mbar_wait_bounded(smem_u32(&bars->empty[stage]), phase ^ 1, p.timeout_ns,
                                           abort_flag, p.status, kSiteProducerEmpty))
                        goto producer_done;
                    const uint32_t rf = smem_u32(&bars->raw_full[stage]);
                    mbar_arrive_expect_tx(rf, RAW_BYTES);
                    tma_load_2d(smem_u32(smem + SmemLayout::raw_off + stage * RAW_STAGE_BYTES),
                                &tmap_w, rf, ks * RAW_ROW, w_row);
                    const uint32_t bf_local = smem_u32(&bars->full[stage]);
                    if (rank == 0) mbar_arrive_expect_tx(bf_local, 2 * ACT_STAGE_BYTES);
#pragma unroll
                    for (int j = 0; j < KPS; ++j)
                        tma_load_2d_pair(smem_u32(smem + SmemLayout::act_off +
                                                  stage * ACT_STAGE_BYTES + j * ACT_BLOCK_BYTES),
                                         &tmap_x, map_to_rank(bf_local, 0), ks * SK + j * BK,
                                         t_row);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:
            // No copy may still be landing, and no MMA-commit arrive from the
            // other CTA may still be in flight, when this CTA exits.
            for (int u = (issued > STAGES ? issued - STAGES : 0); u < issued; ++u) {
                const uint32_t ph = (uint32_t)(u / STAGES) & 1u;
                if (!mbar_wait_drain(smem_u32(&bars->raw_full[u % STAGES]), ph, p.timeout_ns) ||
                    !mbar_wait_drain(smem_u32(&bars->empty[u % STAGES]), ph, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteProducerDrain);
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ------------------------------ MMA issuer (even CTA) -------------
            constexpr uint32_t idesc = idesc_f16_f32acc(2 * BW, BT);
            uint32_t seg_count = 0;
            bool issued_any = false;
            // The issuing thread is on the critical path: each tcgen05.mma
            // costs it ~55 cycles and a k-block's four MMAs run 384 cycles,
            // so the loop keeps to one barrier wait, one four-MMA issue and
            // one commit per k-block, with no division.
            const uint32_t a_base = tmem_base + A_COL0;
            const uint32_t act_base = smem_u32(smem + SmemLayout::act_off);
            uint32_t u = 0;  // k-blocks issued (the ring position)
            WorkIter it(p, cluster, nclusters, num_tiles);
            Work wk;
            if constexpr (GPS == 2) {
                // Whole tiles; stage st holds the groups 2 st and 2 st + 1 (an
                // odd count leaves the last stage's second block, zero-filled
                // by TMA, without a group).
                while (it.next(wk)) {
                    for (int st = wk.kb0; st < wk.kb1; ++st, ++u) {
                        const uint32_t stage = u & (STAGES - 1);
                        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), (u / STAGES) & 1,
                                               p.timeout_ns, abort_flag, p.status, kSiteMmaFull))
                            goto mma_done;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (2 * st + j >= p.G) break;
                            const uint32_t b = seg_count & (NUM_ACC - 1);
                            const uint32_t acc_phase = (seg_count / NUM_ACC) & 1;
                            if (!mbar_wait_bounded(smem_u32(&bars->acc_empty[b]), acc_phase ^ 1,
                                                   p.timeout_ns, abort_flag, p.status,
                                                   kSiteMmaAccEmpty))
                                goto mma_done;
                            tc_fence_after();
                            mma4_pair_a_tmem(
                                tmem_base + b * ACC_COLS,
                                a_base + (u & (A_STAGES - 1)) * A_STAGE_COLS + 32 * j,
                                smem_desc_sw128_kmajor(act_base + stage * ACT_STAGE_BYTES +
                                                       j * ACT_BLOCK_BYTES),
                                idesc, 0u);
                            issued_any = true;
                            tc_commit_pair_multicast(smem_u32(&bars->acc_full[b]), kPairMask);
                            ++seg_count;
                        }
                        tc_commit_pair_multicast(smem_u32(&bars->empty[stage]), kPairMask);
                    }
                }
            }
            while (GPS == 1 && it.next(wk)) {
                int seg_kb, nseg;
                item_segments<MODE, MAX_SEG>(p, wk, seg_kb, nseg);
                (void)nseg;
                for (int kb0 = wk.kb0; kb0 < wk.kb1; kb0 += seg_kb, ++seg_count) {
                    const uint32_t b = seg_count & (NUM_ACC - 1);
                    const uint32_t acc_phase = (seg_count / NUM_ACC) & 1;
                    if (!mbar_wait_bounded(smem_u32(&bars->acc_empty[b]), acc_phase ^ 1,
                                           p.timeout_ns, abort_flag, p.status, kSiteMmaAccEmpty))
                        goto mma_done;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + b * ACC_COLS;
                    const int kb1 = min(wk.kb1, kb0 + seg_kb);
                    for (int kb = kb0; kb < kb1; ++kb, ++u) {
                        const uint32_t stage = u & (STAGES - 1);
                        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), (u / STAGES) & 1,
                                               p.timeout_ns, abort_flag, p.status, kSiteMmaFull))
                            goto mma_done;
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < KPS; ++j)
                            mma4_pair_a_tmem(
                                d_tmem, a_base + (u & (A_STAGES - 1)) * A_STAGE_COLS + 32 * j,
                                smem_desc_sw128_kmajor(act_base + stage * ACT_STAGE_BYTES +
                                                       j * ACT_BLOCK_BYTES),
                                idesc, (kb > kb0 || j > 0) ? 1u : 0u);
                        issued_any = true;
                        // One commit per k-block releases its shared-memory
                        // stage and its A stage on both CTAs.
                        tc_commit_pair_multicast(smem_u32(&bars->empty[stage]), kPairMask);
                    }
                    tc_commit_pair_multicast(smem_u32(&bars->acc_full[b]), kPairMask);
                }
            }
        mma_done:
            if (*abort_flag && issued_any) {
                tc_commit_pair_multicast(smem_u32(&bars->drain), 0x1);
                if (!mbar_wait_drain(smem_u32(&bars->drain), 0, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteDrain);
            }
        }
    } else if (warp < FIRST_EPI_WARP) {
        setmaxnreg_dec<Regs<BITS>::kConv>();
        // ------------------------------ converters (both CTAs) ----------------
        // Thread = weight row r of the CTA's 128 (TMEM lane r): reads its raw
        // k-block (swizzled 16-byte chunks), widens it to 32 fp16 pairs and
        // stores them into the A stage's 32 columns of lane r. Converter
        // warpgroup cg takes the k-blocks u (in the CTA's running order) with
        // u % NUM_CONV_GROUPS == cg, so two k-blocks are widened at once.
        const int q = warp & 3;
        const int cg = (warp - 4) >> 2;
        const int r = q * 32 + lane;
        // The pair's k-blocks, in the order the producer loads them.
        const int total =
            (kStreamK && p.streamk) ? (int)(((int64_t)cluster + 1) * p.units / nclusters -
                              (int64_t)cluster * p.units / nclusters)
                      : ((num_tiles - cluster + nclusters - 1) / nclusters) * p.num_kb;
        for (int u = cg; u < total; u += NUM_CONV_GROUPS) {
            const int stage = u % STAGES, astage = u % A_STAGES;
            const uint32_t phase = (uint32_t)(u / STAGES) & 1u;
            bool ok = mbar_wait_bounded(smem_u32(&bars->raw_full[stage]), phase, p.timeout_ns,
                                        abort_flag, p.status, kSiteConvRaw);
            // A stage u % A_STAGES is free once the MMAs of stage u - A_STAGES
            // completed.
            if (u >= A_STAGES) {
                const int v = u - A_STAGES;
                ok = ok && mbar_wait_bounded(smem_u32(&bars->empty[v % STAGES]),
                                             (uint32_t)(v / STAGES) & 1u, p.timeout_ns,
                                             abort_flag, p.status, kSiteConvA);
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint8_t* raw = smem + SmemLayout::raw_off + stage * RAW_STAGE_BYTES;
            const uint32_t t_a = tmem_base + ((uint32_t)(q * 32) << 16) + A_COL0 +
                                 astage * A_STAGE_COLS;
            // Raw rows of RAW_ROW bytes, swizzled by TMA with a span of RAW_ROW:
            // 16-byte chunk c of row r sits at chunk c ^ ((r >> SH) & (RAW_ROW / 16 - 1)).
            constexpr int SH = RAW_ROW == 128 ? 0 : RAW_ROW == 64 ? 1 : 2;
            const int swz = (r >> SH) & (RAW_ROW / 16 - 1);
#pragma unroll
            for (int h = 0; h < SK / 32; ++h) {  // 32 k per step: 16 columns
                uint32_t v[16];
                if constexpr (BITS == 8) {
                    uint4 w2[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        w2[c] = *reinterpret_cast<const uint4*>(
                            raw + r * RAW_ROW + (((2 * h + c) ^ swz) << 4));
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 w = w2[c];
                        widen_i8x4(w.x, v[8 * c + 0], v[8 * c + 1]);
                        widen_i8x4(w.y, v[8 * c + 2], v[8 * c + 3]);
                        widen_i8x4(w.z, v[8 * c + 4], v[8 * c + 5]);
                        widen_i8x4(w.w, v[8 * c + 6], v[8 * c + 7]);
                    }
                } else {
                    const uint4 w =
                        *reinterpret_cast<const uint4*>(raw + r * RAW_ROW + ((h ^ swz) << 4));
                    widen_i4x8(w.x, v + 0);
                    widen_i4x8(w.y, v + 4);
                    widen_i4x8(w.z, v + 8);
                    widen_i4x8(w.w, v + 12);
                }
                tmem_st_32x32b_x16(t_a + 16 * h, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            // Relaxed arrival: the tensor-memory stores are ordered for the
            // MMA thread by the tcgen05 fences around this synchronization,
            // not by release semantics (a cluster-scope release costs a full
            // memory barrier per k-block).
            if (lane == 0)
                mbar_arrive_cluster_relaxed(map_to_rank(smem_u32(&bars->full[stage]), 0));
        }
    } else {
        setmaxnreg_inc<Regs<BITS>::kEpi>();
        // ------------------------------ epilogue (both CTAs) ------------------
        // Warp w (12..19) owns TMEM lanes 32 * (w % 4).. (32 output channels,
        // one per thread) and the COLS tokens [COLS * half, COLS * half + COLS)
        // of each accumulator, read 32 at a time.
        const int ewarp = warp - FIRST_EPI_WARP;
        const int quad = warp & 3;
        const int half = ewarp >> 2;
        uint8_t* stage_out = smem + SmemLayout::out_off + ewarp * OUT_WARP_BYTES;
        uint32_t seg_count = 0;
        bool store_pending = false;
        bool first_item = true;  // stream-K: partial slot 0 for the first item, 1 after
        uint32_t acc[COLS];

        WorkIter it(p, cluster, nclusters, num_tiles);
        Work wk;
        while (it.next(wk)) {
            int tt, tw;
            tile_coords(p, wk.tile, tt, tw);
            int seg_kb, nseg;
            item_segments<MODE, MAX_SEG>(p, wk, seg_kb, nseg);
            (void)seg_kb;
            const int n_base = tw * (2 * BW) + (int)rank * BW + quad * 32;
            const int n = n_base + lane;                  // this thread's output channel
            const int m_base = tt * BT + half * COLS;     // the warp's first token
            // This thread's scales: per-channel s_w[n], or group g's s_w[n, g]
            // (the next group's prefetched one group ahead).
            float sw_next = 0.0f;
            if (p.s_w != nullptr && n < p.N) sw_next = __ldg(p.s_w + (int64_t)n * p.G);
            if constexpr (MODE == GemmMode::kPgF16) {
#pragma unroll
                for (int j = 0; j < COLS; ++j) acc[j] = 0u;  // f = +0 before the first group
            }
            for (int seg = 0; seg < nseg; ++seg, ++seg_count) {
                const uint32_t b = seg_count % NUM_ACC;
                const uint32_t acc_phase = (seg_count / NUM_ACC) & 1;
                const bool last_seg = (seg == nseg - 1);
                float sw = sw_next;
                if constexpr (MODE == GemmMode::kPgF16) {
                    if (seg + 1 < nseg && n < p.N)
                        sw_next = __ldg(p.s_w + (int64_t)n * p.G + seg + 1);
                }
                {
                    const bool ok = mbar_wait_bounded(smem_u32(&bars->acc_full[b]), acc_phase,
                                                      p.timeout_ns, abort_flag, p.status,
                                                      kSiteEpiAccFull);
                    if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                }
                tc_fence_after();
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       b * ACC_COLS + half * COLS;
                {
                    uint32_t va[LD], vb[LD];
                    tmem_ld_32x32b_x16_ptr(t_row, va);
                    tmem_wait_ld_16(va);
#pragma unroll
                    for (int ch = 0; ch < COLS / LD; ++ch) {
                        uint32_t* v = (ch & 1) ? vb : va;
                        uint32_t* vn = (ch & 1) ? va : vb;
                        if (ch + 1 < COLS / LD) tmem_ld_32x32b_x16_ptr(t_row + (ch + 1) * LD, vn);
                        const int c0 = ch * LD;
                        if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32) {
                            // Exact fp32 integers -> int32: the fast conversion holds
                            // below 2^22; a warp holding a larger one converts all.
                            bool big = false;
#pragma unroll
                            for (int j = 0; j < LD; ++j)
                                big |= fabsf(__uint_as_float(v[j])) >= 4194304.0f;
                            if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                                for (int j = 0; j < LD; ++j) {
                                    const int part = __float2int_rn(__uint_as_float(v[j]));
                                    acc[c0 + j] = (seg == 0) ? (uint32_t)part
                                                             : (uint32_t)((int)acc[c0 + j] + part);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < LD; j += 2) {
                                    float t0, t1;
                                    fadd2_rn(t0, t1, __uint_as_float(v[j]),
                                             __uint_as_float(v[j + 1]), 12582912.0f, 12582912.0f);
                                    const int p0 = __float_as_int(t0) - 0x4B400000;
                                    const int p1 = __float_as_int(t1) - 0x4B400000;
                                    acc[c0 + j] = (seg == 0) ? (uint32_t)p0
                                                             : (uint32_t)((int)acc[c0 + j] + p0);
                                    acc[c0 + j + 1] = (seg == 0)
                                                          ? (uint32_t)p1
                                                          : (uint32_t)((int)acc[c0 + j + 1] + p1);
                                }
                            }
                        } else if constexpr (MODE == GemmMode::kPgF16) {
                            // f = f + fl(P_g * s_g), both roundings kept (ascending
                            // g; f starts at +0). Scalar products: a packed multiply
                            // whose only use is a packed add is contracted into a
                            // fused multiply-add.
#pragma unroll
                            for (int j = 0; j < LD; j += 2) {
                                const float q0 = __fmul_rn(__uint_as_float(v[j]), sw);
                                const float q1 = __fmul_rn(__uint_as_float(v[j + 1]), sw);
                                float r0, r1;
                                fadd2_rn(r0, r1, __uint_as_float(acc[c0 + j]),
                                         __uint_as_float(acc[c0 + j + 1]), q0, q1);
                                acc[c0 + j] = __float_as_uint(r0);
                                acc[c0 + j + 1] = __float_as_uint(r1);
                            }
                        } else {  // kRawPgS32: this group's partials, straight out
                            if (n < p.N) {
#pragma unroll
                                for (int j = 0; j < LD; ++j) {
                                    const int m = m_base + c0 + j;
                                    if (m < p.M)
                                        static_cast<int32_t*>(p.out)[((int64_t)m * p.N + n) * p.G +
                                                                     seg] =
                                            __float2int_rn(__uint_as_float(v[j]));
                                }
                            }
                        }
                        if (ch + 1 < COLS / LD) tmem_wait_ld_16(vn);
                    }
                }
                // This warp's reads of the buffer are complete: release it on
                // the even CTA's barrier (a relaxed arrival: it orders no
                // memory writes).
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster_relaxed(map_to_rank(smem_u32(&bars->acc_empty[b]), 0));

                bool emit = last_seg;
                if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32) {
                    if (kStreamK && last_seg && p.streamk && (wk.kb0 != 0 || wk.kb1 != p.num_kb)) {
                        // A tile shared with other pairs: this CTA's int32
                        // partial, [token][channel] (a warp stores 32
                        // consecutive channels of a token: 128 bytes); the
                        // fix-up launch sums the partials and writes y.
                        const int slot = first_item ? 0 : 1;
                        int32_t* dst = p.part +
                                       ((int64_t)blockIdx.x * 2 + slot) * p.part_rows * BW +
                                       quad * 32 + lane;
#pragma unroll
                        for (int j = 0; j < COLS; ++j) {
                            const int mt = half * COLS + j;  // token within the tile
                            if (mt < p.part_rows) dst[(int64_t)mt * BW] = (int)acc[j];
                        }
                        emit = false;
                    }
                }
                if (emit) {
                    if constexpr (MODE == GemmMode::kRawS32) {
                        if (n < p.N) {
#pragma unroll
                            for (int j = 0; j < COLS; ++j) {
                                const int m = m_base + j;
                                if (m < p.M)
                                    static_cast<int32_t*>(p.out)[(int64_t)m * p.N + n] =
                                        (int)acc[j];
                            }
                        }
                    } else if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kPgF16) {
                        bool big = false;
                        if constexpr (MODE == GemmMode::kPcF16) {
#pragma unroll
                            for (int j = 0; j < COLS; ++j) {
                                const int a = (int)acc[j];
                                big |= (a >= 4194304 || a <= -4194304);
                            }
                        }
                        const bool slow_cvt = __any_sync(0xffffffffu, big);
                        // Rounds of 32 tokens: dequant, stage [token][channel],
                        // TMA store (or direct stores).
#pragma unroll
                        for (int ch = 0; ch < CHUNKS; ++ch) {
                            const int mt = m_base + ch * 32 + lane;  // lane's token of the round
                            const float sa_lane = (mt < p.M) ? __ldg(p.s_a + mt) : 0.0f;
                            uint32_t yv[16];  // token pairs (2j, 2j + 1), 16 bits each
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                const int c = ch * 32 + j;
                                const float sa0 = __shfl_sync(0xffffffffu, sa_lane, j);
                                const float sa1 = __shfl_sync(0xffffffffu, sa_lane, j + 1);
                                float y0, y1;
                                if constexpr (MODE == GemmMode::kPcF16) {
                                    const float f0 = slow_cvt ? __int2float_rn((int)acc[c])
                                                              : small_int_to_float((int)acc[c]);
                                    const float f1 = slow_cvt ? __int2float_rn((int)acc[c + 1])
                                                              : small_int_to_float((int)acc[c + 1]);
                                    float t0, t1;
                                    fmul2_rn(t0, t1, f0, f1, sa0, sa1);
                                    fmul2_rn(y0, y1, t0, t1, sw, sw);
                                } else {
                                    fmul2_rn(y0, y1, __uint_as_float(acc[c]),
                                             __uint_as_float(acc[c + 1]), sa0, sa1);
                                }
                                yv[j / 2] = pack2_rn(y0, y1, p.out_bf16 != 0);
                            }
                            if (p.tma_store) {
                                // The staging buffer is free once the previous
                                // store from it has been read out.
                                if (store_pending && lane == 0) bulk_wait_group_read0();
                                __syncwarp();
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    *reinterpret_cast<uint16_t*>(stage_out + j * 64 + lane * 2) =
                                        (uint16_t)(yv[j / 2] >> (16 * (j & 1)));
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&tmap_y, smem_u32(stage_out), n_base,
                                                 m_base + ch * 32);
                                    bulk_commit_group();
                                }
                                store_pending = true;
                            } else if (n < p.N) {
                                uint16_t* out = static_cast<uint16_t*>(p.out);
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const int m = m_base + ch * 32 + j;
                                    if (m < p.M)
                                        out[(int64_t)m * p.N + n] =
                                            (uint16_t)(yv[j / 2] >> (16 * (j & 1)));
                                }
                            }
                        }
                    }
                }
            }
            first_item = false;
        }
    epi_done:
        // Every output store has completed before the CTA exits.
        if (store_pending && lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA leaves (or frees tensor memory) while the other may still
    // arrive on its barriers or the MMAs may still read or write its tensor
    // memory.
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Stream-K fix-up of the pair kernel (one token tile, tiles_t == 1): every
// weight tile that several pairs shared gets, in each of its two 128-channel
// halves, the sum of the pairs' int32 partials (exact, any order) and the
// per-channel epilogue y = fp16((float(acc) * s_a[m]) * s_w[n]) computed as
// in the GEMM epilogue (or the raw int32 sums). One CTA per 32 tokens x 64
// channels: warp w takes tokens w, w + 8, w + 16, w + 24, lane l channels
// 2 l and 2 l + 1 (8-byte loads; a warp reads and writes whole runs).
// ---------------------------------------------------------------------------
struct FixArgs {
    const int32_t* part;
    int part_rows;
    int64_t units;
    int pairs;  // clusters of the GEMM launch
    int num_kb;
    int M, N;
    const float* s_a;
    const float* s_w;
    void* out;
    int out_bf16;
    int raw_s32;
};

constexpr int FIX_THREADS = 256;
constexpr int FIX_MAX_CONTRIB = kStreamKMaxCtas / 2 + 2;  // pairs sharing one tile
constexpr int64_t kStreamKMinGainKb = 24;

// The stream-K pair whose units include unit u (ranges as in WorkIter).
__device__ __forceinline__ int sk_pair_of_unit(int64_t u, int64_t units, int pairs) {
    return (int)(((u + 1) * pairs + units - 1) / units) - 1;
}

__global__ void __launch_bounds__(FIX_THREADS) sk_fixup_pair_kernel(const FixArgs f) {
    __shared__ const int2* base[FIX_MAX_CONTRIB];  // each contributor's partial half-tile
    grid_dep_wait();
    grid_dep_launch();
    const int chunks = f.part_rows / 32;
    const int half = blockIdx.x & 1;
    const int chunk = (blockIdx.x >> 1) % chunks;
    const int t128 = (blockIdx.x >> 1) / chunks;  // 128-channel tile: pair tile t128 / 2
    const int tw = t128 >> 1, rank = t128 & 1;
    const int64_t u0 = (int64_t)tw * f.num_kb;
    const int p_first = sk_pair_of_unit(u0, f.units, f.pairs);
    const int p_last = sk_pair_of_unit(u0 + f.num_kb - 1, f.units, f.pairs);
    if (p_first == p_last) return;  // one pair did the whole tile and wrote it
    const int nc = p_last - p_first + 1;
    if ((int)threadIdx.x < nc) {
        // The tile is pair c's first item (slot 0) exactly when c's run starts
        // inside it, else its last (slot 1).
        const int c = p_first + (int)threadIdx.x;
        const int64_t c_start = (int64_t)c * f.units / f.pairs;
        const int slot = (c_start / f.num_kb == tw) ? 0 : 1;
        base[threadIdx.x] = reinterpret_cast<const int2*>(
            f.part + ((int64_t)(2 * c + rank) * 2 + slot) * f.part_rows * BW + half * 64);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int acc[4][2] = {};
#pragma unroll 4
    for (int i = 0; i < nc; ++i) {
        int2 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            v[r] = __ldcg(base[i] + (int64_t)(chunk * 32 + warp + 8 * r) * (BW / 2) + lane);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            acc[r][0] += v[r].x;
            acc[r][1] += v[r].y;
        }
    }
    const int n = tw * (2 * BW) + rank * BW + half * 64 + 2 * lane;
    float w0 = 0.0f, w1 = 0.0f;
    if (!f.raw_s32) {
        if (n < f.N) w0 = __ldg(f.s_w + n);
        if (n + 1 < f.N) w1 = __ldg(f.s_w + n + 1);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int m = chunk * 32 + warp + 8 * r;
        if (m >= f.M) break;
        if (f.raw_s32) {
            int32_t* out = static_cast<int32_t*>(f.out) + (int64_t)m * f.N;
            if (n < f.N) out[n] = acc[r][0];
            if (n + 1 < f.N) out[n + 1] = acc[r][1];
        } else {
            const float sa = __ldg(f.s_a + m);
            const uint32_t h = pack2_rn(__fmul_rn(__fmul_rn(__int2float_rn(acc[r][0]), sa), w0),
                                        __fmul_rn(__fmul_rn(__int2float_rn(acc[r][1]), sa), w1),
                                        f.out_bf16 != 0);
            uint16_t* out = static_cast<uint16_t*>(f.out) + (int64_t)m * f.N;
            if (n + 1 < f.N && (f.N & 1) == 0) {
                *reinterpret_cast<uint32_t*>(out + n) = h;
            } else {
                if (n < f.N) out[n] = (uint16_t)(h & 0xFFFFu);
                if (n + 1 < f.N) out[n + 1] = (uint16_t)(h >> 16);
            }
        }
    }
}

}  // namespace gemmw

namespace {

template <GemmMode MODE, int BITS, int BT, int KPS, int GPS = 1>
cudaError_t launch_tw_mode(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty,
                           gemmw::Params p, int32_t* sk_part, int num_sms, cudaStream_t stream) {
    using namespace gemmw;
    using SmemLayout = gemmw::SmemLayout<BT>;
    auto kern = gemm_tw_kernel<MODE, BITS, BT, KPS, GPS>;
    // Once per device: the register count the role split assumes, the
    // shared-memory opt-in, and how many pairs fit on the GPU at once.
    static PerDevice<int> max_clusters_of;
    int max_clusters = 0;
    const cudaError_t e = max_clusters_of.get([&](int& n) {
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemLayout::alloc_bytes);
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = SmemLayout::alloc_bytes;
        cfg.numAttrs = 0;  // the kernel's compile-time cluster shape (2, 1, 1) applies
        r = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (r != cudaSuccess) return r;
        return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
    }, &max_clusters);
    if (e != cudaSuccess) return e;
    const int tiles = p.tiles_t * p.tiles_w;
    int clusters = tiles < max_clusters ? tiles : max_clusters;
    // Stream-K (per-channel, one token tile): every pair takes an equal run of
    // k-blocks, when that shortens the longest pair's run by at least
    // kStreamKMinGainKb k-blocks (the partial stores and the fix-up launch
    // cost about as much as 24 k-blocks of a pair: measured at M = 128, whole
    // tiles win at N10240 K2560, 40 tiles on 74 pairs, 40 against 22
    // k-blocks; stream-K wins at N2560 K10240 and at N28672 K8192).
    // (p.num_kb counts stages of two k-blocks in these kernels.)
    const bool per_channel = (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32);
    const int kps = KPS;
    if (per_channel && sk_part != nullptr && p.tiles_t == 1 && p.num_kb >= 2) {
        const int64_t units = (int64_t)tiles * p.num_kb;
        int g = max_clusters < kStreamKMaxCtas / 2 ? max_clusters : kStreamKMaxCtas / 2;
        if ((int64_t)g > units) g = (int)units;
        const int64_t dp_kb = (int64_t)((tiles + clusters - 1) / clusters) * p.num_kb;
        const int64_t sk_kb = (units + g - 1) / g;
        if ((dp_kb - sk_kb) * kps >= kStreamKMinGainKb) {
            p.streamk = 1;
            p.units = units;
            clusters = g;
            p.part = sk_part;
            p.part_rows = (int)stream_k_part_rows(p.M);
        }
    }
    cudaError_t r = launch_pdl(kern, 2 * clusters, NUM_THREADS, SmemLayout::alloc_bytes, stream,
                               tx, tw, ty, p);
    if (r != cudaSuccess || !p.streamk) return r;
    FixArgs f{};
    f.part = p.part;
    f.part_rows = p.part_rows;
    f.units = p.units;
    f.pairs = clusters;
    f.num_kb = p.num_kb;
    f.M = p.M;
    f.N = p.N;
    f.s_a = p.s_a;
    f.s_w = p.s_w;
    f.out = p.out;
    f.out_bf16 = p.out_bf16;
    f.raw_s32 = (MODE == GemmMode::kRawS32) ? 1 : 0;
    return launch_pdl(sk_fixup_pair_kernel, 2 * tiles * (p.part_rows / 32) * 2, FIX_THREADS, 0,
                      stream, f);
}

}  // namespace

bool gemm_tw_takes_few_tokens(const GemmArgs& a, int num_sms) {
    using namespace gemmw;
    if (a.M > BT_FEW || a.b_raw == nullptr || (a.b_bits != 8 && a.b_bits != 4)) return false;
    if (a.mode == GemmMode::kPcF16) return true;
    if (a.mode != GemmMode::kPgF16) return false;
    // Per group (whole tiles only): when the pairs' tiles occupy at least as
    // many SMs as the single-SM engine's (N = 10240: 80 and 80; N = 2560: 20
    // against 40).
    const int64_t pair_ctas = 2 * std::min<int64_t>((a.N + 2 * BW - 1) / (2 * BW), num_sms / 2);
    const int64_t t128 = (a.N + 127) / 128, t64 = (a.N + 63) / 64;
    const int64_t single_tiles =
        ((t128 + num_sms - 1) / num_sms < (t64 + num_sms - 1) / num_sms) ? t128 : t64;
    return pair_ctas >= std::min<int64_t>(single_tiles, num_sms);
}

cudaError_t launch_gemm_tw(const GemmArgs& a, int num_sms, cudaStream_t stream) {
    using namespace gemmw;
    if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.K % 16 != 0) return cudaErrorInvalidValue;
    if (a.M > INT32_MAX / 2 || a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2)
        return cudaErrorInvalidValue;
    if (!a.b_raw || (a.b_bits != 8 && a.b_bits != 4)) return cudaErrorInvalidValue;
    if (a.b_bits == 4 && a.K % 32 != 0) return cudaErrorInvalidValue;
    const bool per_group = (a.mode == GemmMode::kPgF16 || a.mode == GemmMode::kRawPgS32);
    // Token tile: 128 for at most 128 tokens (one tile), else 192.
    const bool few = a.M <= BT_FEW;
    const int BT = few ? BT_FEW : BT_MANY;
    // k-blocks per stage of the kernel launched: two for the few-token
    // per-channel kernels and for groups of a multiple of 128 k, else one.
    // Per-group layers of 64-k groups take two groups per stage (gps 2);
    // other group sizes that are not a multiple of 128 k keep one k-block
    // per stage.
    const int kps =
        (few && !per_group) ||
                (per_group && (a.group_size == BK || a.group_size % (2 * BK) == 0))
            ? 2
            : 1;
    const int gps = (per_group && a.group_size == BK) ? 2 : 1;
    CUtensorMap tx, tw, ty;
    const uint64_t row_bytes = a.b_bits == 8 ? (uint64_t)a.K : (uint64_t)a.K / 2;
    const uint32_t raw_row = (a.b_bits == 8 ? SK : SK / 2) * kps;  // bytes of one row per stage
    if (encode_tmap_f16_kmajor(&tx, a.a_img, a.M, a.K, BT / 2, BK) != CUDA_SUCCESS ||
        encode_tmap_u8_2d_swizzled(&tw, a.b_raw, a.N, row_bytes, BW,
                                   raw_row, raw_row == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                            : raw_row == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                            : CU_TENSOR_MAP_SWIZZLE_32B) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // 16-bit output through TMA stores of 32 channels x 32 tokens when the
    // row pitch allows it (a multiple of 16 bytes); direct stores otherwise.
    const bool f16_out = (a.mode == GemmMode::kPcF16 || a.mode == GemmMode::kPgF16);
    const bool tma_store = f16_out && (a.N % 8 == 0) &&
                           (reinterpret_cast<uintptr_t>(a.out) % 16 == 0);
    memset(&ty, 0, sizeof(ty));
    if (tma_store && encode_tmap_f16_2d(&ty, a.out, a.M, a.N, 32, 32,
                                        CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    Params p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.bits = a.b_bits;
    p.num_kb = (p.K + BK - 1) / BK;
    if (per_group) {
        if (a.group_size <= 0 || a.group_size % BK != 0 || p.K % a.group_size != 0)
            return cudaErrorInvalidValue;
        if (a.group_size / BK > MAX_SEG_KB) return cudaErrorInvalidValue;  // exact fp32 partials only
        p.num_kb = (p.num_kb + kps - 1) / kps;  // stages
        p.G = p.K / a.group_size;
        // Segments (one per group): whole stages, or half a stage with gps 2.
        p.seg_kb = gps == 2 ? 1 : a.group_size / BK / kps;
    } else {
        // In stages of kps k-blocks; segments of at most MAX_SEG_KB k-blocks.
        p.num_kb = (p.num_kb + kps - 1) / kps;
        const int max_seg = MAX_SEG_KB / kps;
        const int nseg = (p.num_kb + max_seg - 1) / max_seg;
        p.seg_kb = (p.num_kb + nseg - 1) / nseg;
        p.G = 1;
    }
    p.num_seg = gps == 2 ? p.G : (p.num_kb + p.seg_kb - 1) / p.seg_kb;
    p.tiles_t = (p.M + BT - 1) / BT;
    p.tiles_w = (p.N + 2 * BW - 1) / (2 * BW);
    p.w_fastest = (2.0 * (double)p.M > (a.b_bits == 8 ? 1.0 : 0.5) * (double)p.N) ? 1 : 0;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.out = a.out;
    p.tma_store = tma_store ? 1 : 0;
    p.out_bf16 = a.out_bf16;
    p.timeout_ns = a.timeout_ns;
    p.status = a.status;
    // Many tokens: INT8 per-group layers (and their raw int32 test mode); the
    // layer call routes every other layer to the fp16-image pair kernel, which
    // measured faster for them. Few tokens: per-channel (with stream-K) and
    // per-group layers, INT8 or INT4 (gemm_tw_takes_few_tokens).
    if (few) {
        if (a.mode == GemmMode::kPcF16)
            return a.b_bits == 8 ? launch_tw_mode<GemmMode::kPcF16, 8, BT_FEW, 2>(
                                       tx, tw, ty, p, a.sk_part, num_sms, stream)
                                 : launch_tw_mode<GemmMode::kPcF16, 4, BT_FEW, 2>(
                                       tx, tw, ty, p, a.sk_part, num_sms, stream);
        if (a.mode == GemmMode::kPgF16) {
            if (a.b_bits == 8)
                return kps == 1 ? launch_tw_mode<GemmMode::kPgF16, 8, BT_FEW, 1>(
                                      tx, tw, ty, p, nullptr, num_sms, stream)
                       : gps == 2 ? launch_tw_mode<GemmMode::kPgF16, 8, BT_FEW, 2, 2>(
                                        tx, tw, ty, p, nullptr, num_sms, stream)
                                  : launch_tw_mode<GemmMode::kPgF16, 8, BT_FEW, 2>(
                                        tx, tw, ty, p, nullptr, num_sms, stream);
            return kps == 1 ? launch_tw_mode<GemmMode::kPgF16, 4, BT_FEW, 1>(
                                  tx, tw, ty, p, nullptr, num_sms, stream)
                   : gps == 2 ? launch_tw_mode<GemmMode::kPgF16, 4, BT_FEW, 2, 2>(
                                    tx, tw, ty, p, nullptr, num_sms, stream)
                              : launch_tw_mode<GemmMode::kPgF16, 4, BT_FEW, 2>(
                                    tx, tw, ty, p, nullptr, num_sms, stream);
        }
        return cudaErrorInvalidValue;
    }
    if (a.b_bits != 8) return cudaErrorInvalidValue;
    if (a.mode == GemmMode::kPgF16)
        return kps == 1 ? launch_tw_mode<GemmMode::kPgF16, 8, BT_MANY, 1>(tx, tw, ty, p, nullptr,
                                                                          num_sms, stream)
               : gps == 2 ? launch_tw_mode<GemmMode::kPgF16, 8, BT_MANY, 2, 2>(
                                tx, tw, ty, p, nullptr, num_sms, stream)
                          : launch_tw_mode<GemmMode::kPgF16, 8, BT_MANY, 2>(tx, tw, ty, p, nullptr,
                                                                            num_sms, stream);
    if (a.mode == GemmMode::kRawPgS32)
        return kps == 1 ? launch_tw_mode<GemmMode::kRawPgS32, 8, BT_MANY, 1>(
                              tx, tw, ty, p, nullptr, num_sms, stream)
               : gps == 2 ? launch_tw_mode<GemmMode::kRawPgS32, 8, BT_MANY, 2, 2>(
                                tx, tw, ty, p, nullptr, num_sms, stream)
                          : launch_tw_mode<GemmMode::kRawPgS32, 8, BT_MANY, 2>(
                                tx, tw, ty, p, nullptr, num_sms, stream);
    return cudaErrorInvalidValue;
}

}  // namespace cider
