// INT8 x INT8 -> INT32 GEMM with fused dequant on single SMs (cta_group::1
// MMAs): a few-token engine (M <= 128; the layer call takes it for the
// per-group layers whose pair tiles would fill fewer SMs, and for every
// few-token layer under CIDER_GEMM_ENGINE=single), and the tensor-map
// encoders the engines use.
//
// What it computes (Cider README, sections "Metal Kernel Pipeline" and
// "Quantization"): acc[m,n] = sum_k q[m,k] * wq[n,k] exactly in int32, then
//   per-channel: y = fp16(((float)acc * s_a[m]) * s_w[n])            (C = C_int32 * s_act * s_weight)
//   per-group:   f = sum over groups g, ascending, of (float)P_g * s_w[n,g]; y = fp16(f * s_a[m])
// where P_g is the int32 partial over the g-th group of K.
//
// How (B300): tcgen05 has no integer MMA kind on sm_103a, so the codes
// (integers in [-127, 127]) are held exactly as fp16 and multiplied with
// tcgen05.mma kind::f16 into an fp32 accumulator in tensor memory. Every
// product is an integer of magnitude <= 127^2 and every partial sum over at
// most 1024 consecutive k an integer below 127^2 * 1024 < 2^24, exact in
// fp32. K is cut into segments of at most 1024 (per-channel) or of one group
// (per-group); each segment accumulates into one of the TMEM buffers, and
// the epilogue folds it (exact fp32 integer -> int32 and add, or rescale and
// add in fp32 in ascending group order) while the tensor core fills the others.
//
// Shape for few tokens: tiles of 128 tokens x 128 output channels
// (per-channel) or 64 (per-group). With few tokens the weights are nearly
// all of the bytes, so they are read as their raw codes (INT8 [N,K] or
// packed INT4 [N,K/2]) and widened to exact fp16 on chip: TMA stages the raw
// bytes in a deep ring of their own (up to 24 stages) and a warpgroup of
// converter warps writes the 128-byte-swizzled fp16 operand tiles that the
// tensor core reads, in a short ring of operand stages beside the
// activation tiles; no weight image is written to memory. Each stage of both
// rings holds two k-blocks of 64 (one "k-step"), so the MMA thread waits and
// commits once per 128 k. (An fp16 weight image is accepted too, one k-block
// per stage.) Warp 0 issues the raw-code TMA (or, with an image, all of it),
// warp 2 the activation TMA, warp 1 owns TMEM and issues the MMAs
// (128 x BN x 16, the four of a k-block in one go), warps 4-7 convert,
// warps 8-15 are the epilogue: each owns one TMEM lane quadrant and half of
// the tile's columns, reads them 32 at a time, and writes fp16 output
// through 64-byte-swizzled staging and TMA stores. Weight scales are
// fetched by cp.async several segments ahead. Every wait is bounded.
//
// Work split: per-group layers give whole tiles to CTAs (persistent over
// tiles). Per-channel layers use stream-K when it shortens the longest
// CTA's run by at least 12 k-blocks: the tiles' k-steps in tile order are cut
// into one equal run per CTA (80 tiles x 20 k-steps on 148 SMs: 10 or 11
// k-steps each), so a CTA works on the end of one tile and the start of the next;
// a tile shared by several CTAs is stored by each as an exact int32 partial
// and summed, in any order, by a fix-up launch that applies the epilogue.
// Per-group layers cannot be split that way: their result is a rounded fp32
// sum over the groups in ascending order.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {
namespace gemm1 {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;
static_assert(BK == 64, "a k-block is four MMAs of 16 k");
constexpr int MAX_STAGES = 8;       // operand stages (activation + fp16 weight tiles)
constexpr int MAX_RAW_STAGES = 24;  // raw weight-code stages
constexpr int RAW_AB_KB = 4;        // operand k-blocks in flight when the weights arrive raw
// k-blocks per pipeline stage ("k-step"). With raw weight codes a stage holds
// two: the MMA thread waits on a stage's barriers and commits it once per
// 128 k, and that per-stage synchronization, not the tensor core, bounds a
// tile's k loop (an M128 x N128 x K16 MMA takes about 65 cycles, a k-block's
// barrier waits, commit and loop several hundred). fp16 images keep one per
// stage: two would leave fewer than four stages in shared memory.
__host__ __device__ constexpr int stage_kb(int bsrc) { return bsrc != 0 ? 2 : 1; }
// Warps 0-3: TMA producers (warp 0: weight codes, or both operands from an
// image; warp 2: activation tiles when the weights arrive raw), MMA issuer
// and TMEM owner (warp 1); warps 4-7: weight converters (one warpgroup);
// warps 8-15: epilogue.
constexpr int NUM_CONV_WARPS = 4;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int FIRST_EPI_WARP = 8;
constexpr int NUM_THREADS = FIRST_EPI_WARP * 32 + NUM_EPI_THREADS;
constexpr int LAUNCH_REGS = 128;
constexpr int ROLE_REGS = 56;
constexpr int CONV_REGS = 80;
constexpr int EPI_REGS = 184;
static_assert(128 * ROLE_REGS + 128 * CONV_REGS + NUM_EPI_THREADS * EPI_REGS <=
                  NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
constexpr int TMEM_COLS = 512;    // all of TMEM: 512 / BN fp32 accumulators
constexpr int MAX_ACC = 8;
constexpr int MAX_SEG_KB = 16;    // 16 x 64 = 1024 k per exact fp32 segment
constexpr int OUT_WARP_BYTES = 32 * 32 * 2;  // one 32 x 32 fp16 store box per warp
constexpr int SMEM_LIMIT = 232448;           // opt-in shared memory per block

// Groups per TMEM buffer: per-group tiles of 64 columns hold 4, of 128
// columns 2 (two buffers of 256 columns); per-channel tiles 1.
__host__ __device__ constexpr int tile_groups(GemmMode mode, int bn) {
    return (mode == GemmMode::kPgF16 || mode == GemmMode::kRawPgS32) ? (bn == 64 ? 4 : 2) : 1;
}

// Per-instantiation shape. BSRC: weight operand source, 0 = fp16 image (TMA
// straight into the operand tile), 8 / 4 = raw INT8 / packed INT4 codes
// widened on chip. BN: tile width in output channels. An MMA of M128 x N64
// holds the issuing thread almost as long as one of N128 (56 against 65
// cycles on B300), so per-channel tiles are 128 wide; per-group tiles are
// 128 or 64 wide (the launcher's wave rule).
template <int BSRC, int BN, int GROUPS>
struct Cfg {
    static constexpr bool kRaw = BSRC != 0;
    static constexpr int kKps = stage_kb(BSRC);  // k-blocks per stage
    static constexpr int kCols = BN / 2;        // columns per epilogue warp
    static constexpr int kChunks = kCols / 32;  // 32-column TMEM loads per warp and segment
    // Per-group tiles hold kGroups groups' partials side by side in one TMEM
    // buffer (one accumulator of BN columns per group), so the tensor core and
    // the epilogue hand over once per kGroups groups, not once per group.
    static constexpr int kGroups = GROUPS;
    static constexpr int kBufCols = kGroups * BN;
    static constexpr int kNumAcc = TMEM_COLS / kBufCols;
    static constexpr int kScaleDepth = 2;  // scale sets (one per segment) in flight per warp
    // A stage holds kKps k-blocks: activation tiles of A_STAGE_BYTES and fp16
    // weight tiles of kBBlockBytes, each block's tile a whole swizzled operand.
    static constexpr int kAStageBytes = kKps * A_STAGE_BYTES;
    static constexpr int kBBlockBytes = BN * BK * 2;
    static constexpr int kBStageBytes = kKps * kBBlockBytes;
    // Raw codes of one row and k-block; a raw stage holds the kKps blocks one
    // after the other, each BN rows of kRawRowBytes (the converters' reads of
    // a block then cover contiguous bytes, free of bank conflicts).
    static constexpr int kRawRowBytes = BSRC == 8 ? BK : BK / 2;
    static constexpr int kRawBlockBytes = kRaw ? BN * kRawRowBytes : 0;
    static constexpr int kRawBytes = kKps * kRawBlockBytes;
    static constexpr int kFullTx = kRaw ? kAStageBytes : kAStageBytes + kBStageBytes;
    static constexpr int kScaleFloats = kScaleDepth * kGroups * kCols;  // per epilogue warp
    static constexpr int kFixedBytes = NUM_EPI_WARPS * OUT_WARP_BYTES +
                                       NUM_EPI_WARPS * kScaleFloats * 4 + 1024 + 16 + 1024;
    static constexpr int kABBytes = kAStageBytes + kBStageBytes;
    static constexpr int kAvail = SMEM_LIMIT - kFixedBytes;
    // Image weights: one ring of operand stages, as deep as fits. Raw codes:
    // the operand ring stays short (its tiles come from L2 or are written on
    // chip) and the rest of shared memory holds raw-code stages, so that
    // enough weight bytes are in flight from HBM per SM; with one ring for
    // everything (five stages) a few-token layer ran at a fixed number of
    // microseconds per k-block whatever the code width or token count.
    static constexpr int kStages = kRaw ? RAW_AB_KB / kKps
                                        : (kAvail / kABBytes < MAX_STAGES ? kAvail / kABBytes
                                                                          : MAX_STAGES);
    static constexpr int kRawFit = kRaw ? (kAvail - kStages * kABBytes) / kRawBytes : 0;
    static constexpr int kRawStages = kRawFit < MAX_RAW_STAGES ? kRawFit : MAX_RAW_STAGES;
    static_assert(kNumAcc >= 2 && kNumAcc <= MAX_ACC && kChunks >= 1, "tile width");
    static_assert(kStages >= 2 && kStages * kKps >= 4, "pipeline depth");
    static_assert(!kRaw || kRawStages >= 4, "raw pipeline depth");
    static_assert(kRaw || kKps == 1, "image operands stage one k-block");
};

struct __align__(8) Barriers {
    uint64_t full[MAX_STAGES];       // TMA of the activation (and image weight) tiles
    uint64_t conv_full[MAX_STAGES];  // converters wrote the fp16 weight tile
    uint64_t empty[MAX_STAGES];      // the MMAs reading the stage completed
    uint64_t raw_full[MAX_RAW_STAGES];   // TMA of a raw weight tile
    uint64_t raw_empty[MAX_RAW_STAGES];  // the converters took the raw tile into registers
    uint64_t acc_full[MAX_ACC];
    uint64_t acc_empty[MAX_ACC];
    uint64_t drain;
};
static_assert(sizeof(Barriers) <= 1024, "barrier area");

template <int BSRC, int BN, int GROUPS>
struct SmemLayout {
    using C = Cfg<BSRC, BN, GROUPS>;
    static constexpr int STAGES = C::kStages;
    static constexpr int RAW_STAGES = C::kRawStages;
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + STAGES * C::kAStageBytes;
    static constexpr int raw_off = b_off + STAGES * C::kBStageBytes;
    static constexpr int out_off = raw_off + RAW_STAGES * C::kRawBytes;
    static constexpr int scale_off = out_off + NUM_EPI_WARPS * OUT_WARP_BYTES;
    static constexpr int bar_off = scale_off + NUM_EPI_WARPS * C::kScaleFloats * 4;
    static constexpr int misc_off = bar_off + 1024;  // tmem base, abort
    static constexpr int bytes = misc_off + 16;
    static constexpr int alloc_bytes = bytes + 1024;  // runtime 1024-byte alignment slack
    static_assert(alloc_bytes <= SMEM_LIMIT, "shared memory per block");
    static_assert(out_off % 1024 == 0, "64-byte-swizzled staging alignment");
};

struct Params {
    int M, N, K;
    int num_kb;   // k-steps (stages of stage_kb(BSRC) k-blocks of 64) per tile
    int num_blk;  // k-blocks of 64 (the last k-step may hold one block past K)
    int seg_kb;   // k-steps per segment
    int num_seg;  // segments per tile
    int group_kb; // k-blocks per group (per-group; MAX_SEG_KB, no split, per-channel)
    int G;        // columns of s_w (1 for per-channel)
    int tiles_m, tiles_n;
    const float* s_a;
    const float* s_w;
    const float* s_wT;  // group-major copy of per-group s_w, or NULL
    void* out;
    int tma_store;  // fp16 output written through tmap_y (N % 8 == 0)
    int out_bf16;   // output elements are bfloat16 instead of fp16
    uint64_t timeout_ns;
    unsigned long long* status;
    // Stream-K (per-channel modes): the tiles' num_kb-long k-step runs form
    // `units` units, CTA c takes units [c * units / grid, (c + 1) * units /
    // grid). A tile that several CTAs share is left to the fix-up kernel:
    // each stores its int32 partial of the tile in `part`.
    int streamk;
    int64_t units;
    int32_t* part;  // [grid][2][BN / 4][part_rows][4] int32
    int part_rows;
};

// Wait sites recorded in the device status word on a timeout.
enum : uint32_t {
    kSiteProducerEmpty = 0x101,
    kSiteMmaAccEmpty = 0x102,
    kSiteMmaFull = 0x103,
    kSiteEpiAccFull = 0x104,
    kSiteDrain = 0x105,
    kSiteProducerDrain = 0x106,
    kSiteConvRaw = 0x107,
    kSiteMmaConv = 0x108,
    kSiteConvEmpty = 0x109,
};

// A CTA's work item: k-steps [kb0, kb1) of one tile.
struct Work {
    int tile, kb0, kb1;
};

// The items of this CTA, in order: whole tiles blockIdx.x, + gridDim.x, ...;
// or with stream-K its run of units, cut at tile boundaries.
struct WorkIter {
    int64_t u, uend;
    int tile, num_tiles, nk;
    bool sk;
    __device__ __forceinline__ WorkIter(const Params& p, int num_tiles_)
        : tile((int)blockIdx.x), num_tiles(num_tiles_), nk(p.num_kb), sk(p.streamk != 0) {
        u = sk ? (int64_t)blockIdx.x * p.units / gridDim.x : 0;
        uend = sk ? ((int64_t)blockIdx.x + 1) * p.units / gridDim.x : 0;
    }
    __device__ __forceinline__ bool next(Work& w) {
        if (sk) {
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
        tile += gridDim.x;
        return true;
    }
};

// The stream-K CTA whose units include unit u (ranges as in WorkIter).
__device__ __forceinline__ int sk_cta_of_unit(int64_t u, int64_t units, int grid) {
    return (int)(((u + 1) * grid + units - 1) / units) - 1;
}

// Segments of an item: per-group, the tile's fixed segments (items are whole
// tiles); per-channel, the item's k-steps in equal runs of at most
// MAX_SEG_KB k-blocks.
template <GemmMode MODE, int KPS>
__device__ __forceinline__ void item_segments(const Params& p, const Work& w, int& seg_kb,
                                              int& nseg) {
    if constexpr (MODE == GemmMode::kPgF16 || MODE == GemmMode::kRawPgS32) {
        seg_kb = p.seg_kb;
        nseg = p.num_seg;
    } else {
        constexpr int MAX_SEG = MAX_SEG_KB / KPS;
        const int len = w.kb1 - w.kb0;
        const int n = (len + MAX_SEG - 1) / MAX_SEG;
        seg_kb = (len + n - 1) / n;
        nseg = (len + seg_kb - 1) / seg_kb;
    }
}

// The four MMAs of one k-block (4 x 16 k; both operands advance 32 bytes
// within their 128-byte swizzle rows, 2 in descriptor units), issued from one
// asm block; the first accumulates only if `accumulate`.
__device__ __forceinline__ void mma4_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, t;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"(a_desc + 2), "l"(b_desc + 2),
        "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
        : "memory");
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int& tm, int& tn) {
    tm = tile % tiles_m;
    tn = tile / tiles_m;
}

// Widens one 16-byte piece of raw weight codes (INT8: 16 codes; packed INT4:
// 32 codes) of operand row r, starting at 16-byte chunk c0 of the fp16 row
// (8 codes per chunk), into the 128-byte-swizzled K-major tile: chunk c of
// row r lives at byte r * 128 + ((c ^ (r & 7)) << 4). Each code u-shifted to
// [0, 256) becomes the fp16 1024 + u by placing u under the exponent byte
// 0x64, and an exact fp16 subtraction removes the offset.
template <int BSRC>
__device__ __forceinline__ void widen_piece(const uint4 raw, uint8_t* tile, int r, int c0) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    constexpr int NH = (BSRC == 8) ? 8 : 16;  // fp16 pairs produced
    uint32_t h[NH];
    if constexpr (BSRC == 8) {
        const __half2 bias = __float2half2_rn(1152.0f);  // 1024 + 128
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t u = w[i] ^ 0x80808080u;  // signed byte b -> b + 128
            const uint32_t t0 = __byte_perm(u, 0x64646464u, 0x5140);  // codes 4i, 4i+1
            const uint32_t t1 = __byte_perm(u, 0x64646464u, 0x7362);  // codes 4i+2, 4i+3
            __half2 v0 = __hsub2(*reinterpret_cast<const __half2*>(&t0), bias);
            __half2 v1 = __hsub2(*reinterpret_cast<const __half2*>(&t1), bias);
            h[2 * i] = *reinterpret_cast<uint32_t*>(&v0);
            h[2 * i + 1] = *reinterpret_cast<uint32_t*>(&v1);
        }
    } else {
        // Nibble = code + 8; element 2j is the low nibble of byte j.
        const __half2 bias = __float2half2_rn(1032.0f);  // 1024 + 8
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = w[i] & 0x0F0F0F0Fu;            // elements 8i, 8i+2, 8i+4, 8i+6
            const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;     // elements 8i+1, 8i+3, ...
            const uint32_t e0 = __byte_perm(lo, hi, 0x5140);   // elements 8i .. 8i+3
            const uint32_t e1 = __byte_perm(lo, hi, 0x7362);   // elements 8i+4 .. 8i+7
            const uint32_t t[4] = {__byte_perm(e0, 0x64646464u, 0x5140),
                                   __byte_perm(e0, 0x64646464u, 0x7362),
                                   __byte_perm(e1, 0x64646464u, 0x5140),
                                   __byte_perm(e1, 0x64646464u, 0x7362)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&t[j]), bias);
                h[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NH / 4; ++q)
        *reinterpret_cast<uint4*>(tile + r * 128 + (((c0 + q) ^ (r & 7)) << 4)) =
            make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
}

template <GemmMode MODE, int BSRC, int BN>
__global__ void __maxnreg__(LAUNCH_REGS)
    gemm_tc1_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_y, const Params p) {
    constexpr int GROUPS_ = tile_groups(MODE, BN);
    using Layout = SmemLayout<BSRC, BN, GROUPS_>;
    using C = Cfg<BSRC, BN, GROUPS_>;
    constexpr int STAGES = Layout::STAGES;
    constexpr int RAW_STAGES = Layout::RAW_STAGES > 0 ? Layout::RAW_STAGES : 1;
    constexpr int KPS = C::kKps;
    constexpr int NUM_ACC = C::kNumAcc;
    constexpr int COLS = C::kCols;
    constexpr int SD = C::kScaleDepth;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bars = reinterpret_cast<Barriers*>(smem + Layout::bar_off);
    float* scales = reinterpret_cast<float*>(smem + Layout::scale_off);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + Layout::misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Layout::misc_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.tiles_m * p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->conv_full[s]), NUM_CONV_WARPS);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int r = 0; r < RAW_STAGES; ++r) {
            mbar_init(smem_u32(&bars->raw_full[r]), 1);
            mbar_init(smem_u32(&bars->raw_empty[r]), NUM_CONV_WARPS);
        }
        for (int b = 0; b < NUM_ACC; ++b) {
            mbar_init(smem_u32(&bars->acc_full[b]), 1);
            mbar_init(smem_u32(&bars->acc_empty[b]), NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        if (p.tma_store) prefetch_tmap(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_base_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_slot;
    // Everything above overlaps the tail of the preceding kernel (programmatic
    // dependent launch); global memory is touched only after this wait.
    grid_dep_wait();
    grid_dep_launch();

    if (warp < 4) setmaxnreg_dec<ROLE_REGS>();
    if ((C::kRaw ? warp == 2 : warp == 0) && lane == 0) {
        // -------------------- TMA producer: operand stages --------------------
        // The activation tiles of each k-step's k-blocks, and with an image
        // their fp16 weight tiles too, into the operand stage its MMAs read (a
        // block past K reads as zeros).
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        WorkIter it(p, num_tiles);
        Work w;
        while (it.next(w)) {
            int tm, tn;
            tile_coords(w.tile, p.tiles_m, tm, tn);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&bars->empty[stage]), phase ^ 1, p.timeout_ns,
                                       abort_flag, p.status, kSiteProducerEmpty))
                    goto producer_done;
                const uint32_t fb = smem_u32(&bars->full[stage]);
                mbar_arrive_expect_tx(fb, C::kFullTx);
#pragma unroll
                for (int j = 0; j < KPS; ++j) {
                    tma_load_2d(smem_u32(smem + Layout::a_off + stage * C::kAStageBytes +
                                         j * A_STAGE_BYTES),
                                &tmap_a, fb, (kb * KPS + j) * BK, tm * BM);
                    if constexpr (!C::kRaw)
                        tma_load_2d(smem_u32(smem + Layout::b_off + stage * C::kBStageBytes +
                                             j * C::kBBlockBytes),
                                    &tmap_b, fb, (kb * KPS + j) * BK, tn * BN);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    producer_done:
        if (*abort_flag) {
            // Let every load already issued land before the CTA exits: the
            // last use u of each stage completes phase u / STAGES.
            for (int u = (issued > STAGES ? issued - STAGES : 0); u < issued; ++u) {
                const uint32_t par = (uint32_t)(u / STAGES) & 1u;
                if (!mbar_wait_drain(smem_u32(&bars->full[u % STAGES]), par, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteProducerDrain);
            }
        }
    } else if (C::kRaw && warp == 0 && lane == 0) {
        // -------------------- TMA producer: raw weight codes -----------------
        // Runs up to RAW_STAGES k-steps ahead of the converters; one box per
        // k-block of the k-step, BN rows each.
        int rstage = 0;
        uint32_t rphase = 0;
        int issued = 0;
        WorkIter it(p, num_tiles);
        Work w;
        while (it.next(w)) {
            int tm, tn;
            tile_coords(w.tile, p.tiles_m, tm, tn);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait_bounded(smem_u32(&bars->raw_empty[rstage]), rphase ^ 1,
                                       p.timeout_ns, abort_flag, p.status, kSiteProducerEmpty))
                    goto raw_producer_done;
                const uint32_t rb = smem_u32(&bars->raw_full[rstage]);
                mbar_arrive_expect_tx(rb, C::kRawBytes);
#pragma unroll
                for (int j = 0; j < KPS; ++j)
                    tma_load_2d(smem_u32(smem + Layout::raw_off + rstage * C::kRawBytes +
                                         j * C::kRawBlockBytes),
                                &tmap_b, rb, (kb * KPS + j) * C::kRawRowBytes, tn * BN);
                ++issued;
                if (++rstage == RAW_STAGES) {
                    rstage = 0;
                    rphase ^= 1;
                }
            }
        }
    raw_producer_done:
        if (*abort_flag) {
            for (int u = (issued > RAW_STAGES ? issued - RAW_STAGES : 0); u < issued; ++u) {
                const uint32_t par = (uint32_t)(u / RAW_STAGES) & 1u;
                if (!mbar_wait_drain(smem_u32(&bars->raw_full[u % RAW_STAGES]), par,
                                     p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteProducerDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32acc(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t seg_count = 0;
            bool issued_any = false;
            WorkIter it(p, num_tiles);
            Work w;
            while (it.next(w)) {
                int seg_kb, nseg;
                item_segments<MODE, KPS>(p, w, seg_kb, nseg);
                for (int seg = 0; seg < nseg; ++seg, ++seg_count) {
                    const uint32_t b = seg_count % NUM_ACC;
                    const uint32_t acc_phase = (seg_count / NUM_ACC) & 1;
                    if (!mbar_wait_bounded(smem_u32(&bars->acc_empty[b]), acc_phase ^ 1,
                                           p.timeout_ns, abort_flag, p.status, kSiteMmaAccEmpty))
                        goto mma_done;
                    tc_fence_after();
                    const int kb0 = w.kb0 + seg * seg_kb;
                    const int kb1 = min(w.kb1, kb0 + seg_kb);
                    // Group j of the segment accumulates into its own BN
                    // columns; gpos is the k-block's position in its group
                    // (segments start on group boundaries, and a group may
                    // end inside a k-step).
                    uint32_t d_tmem = tmem_base + b * C::kBufCols;
                    int gpos = 0;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), phase, p.timeout_ns,
                                               abort_flag, p.status, kSiteMmaFull))
                            goto mma_done;
                        if (C::kRaw &&
                            !mbar_wait_bounded(smem_u32(&bars->conv_full[stage]), phase,
                                               p.timeout_ns, abort_flag, p.status, kSiteMmaConv))
                            goto mma_done;
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < KPS; ++j) {
                            if (KPS == 1 || kb * KPS + j < p.num_blk) {
                                mma4_f16(d_tmem,
                                         smem_desc_sw128_kmajor(smem_u32(
                                             smem + Layout::a_off + stage * C::kAStageBytes +
                                             j * A_STAGE_BYTES)),
                                         smem_desc_sw128_kmajor(smem_u32(
                                             smem + Layout::b_off + stage * C::kBStageBytes +
                                             j * C::kBBlockBytes)),
                                         idesc, gpos > 0 ? 1u : 0u);
                                if (++gpos == p.group_kb) {
                                    gpos = 0;
                                    d_tmem += BN;
                                }
                            }
                        }
                        issued_any = true;
                        tc_commit(smem_u32(&bars->empty[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    tc_commit(smem_u32(&bars->acc_full[b]));
                }
            }
        mma_done:
            if (*abort_flag && issued_any) {
                // Every MMA issued so far must finish before TMEM is released.
                tc_commit(smem_u32(&bars->drain));
                if (!mbar_wait_drain(smem_u32(&bars->drain), 0, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteDrain);
            }
        }
    } else if (warp < 4) {
        // idle role warps
    } else if (warp < FIRST_EPI_WARP) {
        setmaxnreg_dec<CONV_REGS>();
        // ------------------------- weight converters --------------------------
        // Block j of a raw stage is BN rows of kRawRowBytes, i.e. PPK 16-byte
        // pieces per row, widened into its own fp16 operand tile: its piece
        // pc covers row pc / PPK, fp16 chunks from (pc % PPK) * CPP.
        if constexpr (C::kRaw) {
            constexpr int PPK = C::kRawRowBytes / 16;
            constexpr int CPP = 8 / PPK;
            constexpr int PER_THREAD = BN * PPK / (32 * NUM_CONV_WARPS);
            static_assert(CPP * PPK == 8, "raw pieces per k-block");
            static_assert(PER_THREAD >= 1 && PER_THREAD * 32 * NUM_CONV_WARPS == BN * PPK,
                          "converter work split");
            const int ct = (warp - 4) * 32 + lane;
            int stage = 0, rstage = 0;
            uint32_t phase = 0, rphase = 0;
            WorkIter it(p, num_tiles);
            Work w;
            while (it.next(w)) {
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    {
                        const bool ok = mbar_wait_bounded(smem_u32(&bars->raw_full[rstage]),
                                                          rphase, p.timeout_ns, abort_flag,
                                                          p.status, kSiteConvRaw);
                        if (!__all_sync(0xffffffffu, ok)) goto conv_done;
                    }
                    const uint4* raw = reinterpret_cast<const uint4*>(
                        smem + Layout::raw_off + rstage * C::kRawBytes);
#pragma unroll
                    for (int j = 0; j < KPS; ++j) {
                        uint8_t* tile_b =
                            smem + Layout::b_off + stage * C::kBStageBytes + j * C::kBBlockBytes;
                        uint4 pcs[PER_THREAD];
#pragma unroll
                        for (int i = 0; i < PER_THREAD; ++i) {
                            const int pc = ct + i * 32 * NUM_CONV_WARPS;
                            pcs[i] = raw[j * (BN * PPK) + pc];
                        }
                        if (j == 0) {
                            // The fp16 tiles of this operand stage are free once
                            // the MMAs of its previous k-step completed.
                            const bool ok =
                                mbar_wait_bounded(smem_u32(&bars->empty[stage]), phase ^ 1,
                                                  p.timeout_ns, abort_flag, p.status,
                                                  kSiteConvEmpty);
                            if (!__all_sync(0xffffffffu, ok)) goto conv_done;
                        }
#pragma unroll
                        for (int i = 0; i < PER_THREAD; ++i) {
                            const int pc = ct + i * 32 * NUM_CONV_WARPS;
                            widen_piece<BSRC>(pcs[i], tile_b, pc / PPK, (pc % PPK) * CPP);
                        }
                    }
                    // Order this warp's generic-proxy accesses before the
                    // async proxy's: its fp16 writes before the tensor core's
                    // reads, its reads of the raw stage (consumed above) before
                    // the next copy into it. Then release both stages.
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bars->raw_empty[rstage]));
                        mbar_arrive(smem_u32(&bars->conv_full[stage]));
                    }
                    if (++rstage == RAW_STAGES) {
                        rstage = 0;
                        rphase ^= 1;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        conv_done:;
        }
    } else {
        setmaxnreg_inc<EPI_REGS>();
        // ------------------------------ epilogue ------------------------------
        // Warp w (8..15) owns TMEM lanes 32 * (w % 4) .. +31 (its 32 token
        // rows; a warp may only access its own lane quadrant) and the COLS
        // columns [COLS * half, COLS * half + COLS) of the tile, read 32 at a
        // time.
        const int ewarp = warp - FIRST_EPI_WARP;
        const int quad = warp & 3;
        const int half = ewarp >> 2;
        uint8_t* stage_out = smem + Layout::out_off + ewarp * OUT_WARP_BYTES;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);  // 64-byte swizzle of row `lane`
        // Weight scales, SD sets per warp in flight: a "use" is one segment
        // (per-group: the scales of its kGroups groups) or the last segment of
        // a tile (per-channel); lanes copy their columns with cp.async, one
        // commit group per use, SD - 1 uses ahead of the one being folded.
        constexpr bool kPerSegScales = (MODE == GemmMode::kPgF16);
        constexpr int GS = C::kGroups;
        constexpr int SET = GS * COLS;  // floats per use: [group][column]
        float* wsc = scales + ewarp * C::kScaleFloats;
        // Next use to fetch: item fw, segment f_seg of it (per-group).
        WorkIter f_it(p, num_tiles);
        Work fw;
        bool f_ok = f_it.next(fw);
        int f_seg = 0;
        uint32_t f_slot = 0, u_slot = 0;
        auto fetch_next = [&]() {
            if (f_ok) {
                int tm, tn;
                tile_coords(fw.tile, p.tiles_m, tm, tn);
                float* dst = wsc + f_slot * SET;
#pragma unroll
                for (int j = 0; j < GS; ++j) {
                    const int g = (p.G == 1) ? 0 : f_seg * GS + j;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        const int n = tn * BN + half * COLS + c * 32 + lane;
                        float* d = dst + j * COLS + c * 32 + lane;
                        if (p.s_w != nullptr && n < p.N && g < p.G) {
                            const float* src = (p.s_wT != nullptr) ? p.s_wT + (int64_t)g * p.N + n
                                                                   : p.s_w + (int64_t)n * p.G + g;
                            cp_async_4(smem_u32(d), src);
                        } else {
                            *d = 0.0f;
                        }
                    }
                }
                if (kPerSegScales && f_seg + 1 < p.num_seg) {
                    ++f_seg;
                } else {
                    f_seg = 0;
                    f_ok = f_it.next(fw);
                }
            }
            cp_async_commit();  // possibly empty: one group per use keeps the count
            f_slot = (f_slot + 1 == SD) ? 0 : f_slot + 1;
        };
        for (int i = 0; i < SD - 1; ++i) fetch_next();
        uint32_t seg_count = 0;
        bool store_pending = false;
        uint32_t acc[COLS];  // int32 running sum (per-channel) or fp32 running sum (per-group)
        bool first_item = true;  // stream-K: partial slot 0 for the first item, 1 after

        WorkIter it(p, num_tiles);
        Work w;
        while (it.next(w)) {
            int tm, tn;
            tile_coords(w.tile, p.tiles_m, tm, tn);
            const int m_base = tm * BM + quad * 32;
            const int m = m_base + lane;
            const int n_w = tn * BN + half * COLS;
            int seg_kb, nseg;
            item_segments<MODE, KPS>(p, w, seg_kb, nseg);
            (void)seg_kb;
            if constexpr (MODE == GemmMode::kPgF16) {
#pragma unroll
                for (int j = 0; j < COLS; ++j) acc[j] = 0u;  // f = +0 before the first group
            }
            for (int seg = 0; seg < nseg; ++seg, ++seg_count) {
                const uint32_t b = seg_count % NUM_ACC;
                const uint32_t acc_phase = (seg_count / NUM_ACC) & 1;
                const bool last_seg = (seg == nseg - 1);
                const bool uses_scales = kPerSegScales || last_seg;
                const float* sc = wsc + u_slot * SET;
                if (uses_scales) {
                    __syncwarp();  // every lane is done reading the slot refilled next
                    fetch_next();
                    cp_async_wait_group<SD - 1>();  // this use's group has landed
                    __syncwarp();
                }
                {
                    // Every lane waits; the warp leaves together if any lane gave
                    // up, so the warp-wide tcgen05.ld is always issued by all lanes.
                    const bool ok = mbar_wait_bounded(smem_u32(&bars->acc_full[b]), acc_phase,
                                                      p.timeout_ns, abort_flag, p.status,
                                                      kSiteEpiAccFull);
                    if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                }
                tc_fence_after();
                {
                  // Groups of this segment (per-group), in ascending order.
                  const int ng = (MODE == GemmMode::kPgF16 || MODE == GemmMode::kRawPgS32)
                                     ? min(GS, p.G - seg * GS)
                                     : 1;
                  for (int j = 0; j < ng; ++j) {  // warp-uniform
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32_ptr(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                               b * C::kBufCols + j * BN + half * COLS + c * 32,
                                           v);
                    tmem_wait_ld_32(v);
                    uint32_t* ac = acc + c * 32;
                    if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32) {
                        // Exact fp32 integers -> int32 (the short conversion is exact
                        // below 2^22; the warp takes the long one if any lane needs it).
                        bool big = false;
#pragma unroll
                        for (int i = 0; i < 32; ++i) big |= fabsf(__uint_as_float(v[i])) >= 4194304.0f;
                        if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int part = __float2int_rn(__uint_as_float(v[i]));
                                ac[i] = (seg == 0) ? (uint32_t)part : (uint32_t)((int)ac[i] + part);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int part = small_float_to_int(__uint_as_float(v[i]));
                                ac[i] = (seg == 0) ? (uint32_t)part : (uint32_t)((int)ac[i] + part);
                            }
                        }
                    } else if constexpr (MODE == GemmMode::kPgF16) {
                        // f = f + fl(P_g * s_g): scalar products (a packed product
                        // whose only use is a packed add is fused), packed adds.
                        const float* scc = sc + j * COLS + c * 32;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 s4 = *reinterpret_cast<const float4*>(scc + i);
                            const float q0 = __fmul_rn(__uint_as_float(v[i]), s4.x);
                            const float q1 = __fmul_rn(__uint_as_float(v[i + 1]), s4.y);
                            const float q2 = __fmul_rn(__uint_as_float(v[i + 2]), s4.z);
                            const float q3 = __fmul_rn(__uint_as_float(v[i + 3]), s4.w);
                            float r0, r1, r2, r3;
                            fadd2_rn(r0, r1, __uint_as_float(ac[i]), __uint_as_float(ac[i + 1]),
                                     q0, q1);
                            fadd2_rn(r2, r3, __uint_as_float(ac[i + 2]),
                                     __uint_as_float(ac[i + 3]), q2, q3);
                            ac[i] = __float_as_uint(r0);
                            ac[i + 1] = __float_as_uint(r1);
                            ac[i + 2] = __float_as_uint(r2);
                            ac[i + 3] = __float_as_uint(r3);
                        }
                    } else {  // kRawPgS32: this group's partials, written directly
                        const int n_c = n_w + c * 32;
                        if (m < p.M && n_c < p.N) {
                            int32_t* out = static_cast<int32_t*>(p.out) +
                                           ((int64_t)m * p.N + n_c) * p.G + seg * GS + j;
                            const int valid = min(32, p.N - n_c);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < valid)
                                    out[(int64_t)i * p.G] = __float2int_rn(__uint_as_float(v[i]));
                        }
                    }
                    }
                  }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[b]));

                bool emit = last_seg;
                if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32) {
                    if (last_seg && p.streamk && (w.kb0 != 0 || w.kb1 != p.num_kb)) {
                        // ---- stream-K: a tile shared with other CTAs ----
                        // Only this CTA's int32 partial of its rows and columns
                        // is stored; the fix-up kernel sums the partials and
                        // writes the output. A partial tile is [BN / 4]
                        // [part_rows] runs of four columns, so that the 32 lanes
                        // (32 rows) of a warp store 512 contiguous bytes.
                        const int r = quad * 32 + lane;
                        const int slot = first_item ? 0 : 1;
                        if (r < p.part_rows) {
                            int4* dst = reinterpret_cast<int4*>(p.part) +
                                        (((int64_t)blockIdx.x * 2 + slot) * (BN / 4) +
                                         half * (COLS / 4)) * p.part_rows + r;
#pragma unroll
                            for (int j = 0; j < COLS; j += 4)
                                dst[(j / 4) * p.part_rows] =
                                    make_int4((int)acc[j], (int)acc[j + 1], (int)acc[j + 2],
                                              (int)acc[j + 3]);
                        }
                        emit = false;
                    }
                }
                if (emit) {
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        const uint32_t* ac = acc + c * 32;
                        const int n_c = n_w + c * 32;
                        if constexpr (MODE == GemmMode::kRawS32) {
                            if (m < p.M) {
                                int32_t* out = static_cast<int32_t*>(p.out) + (int64_t)m * p.N;
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (n_c + j < p.N) out[n_c + j] = (int)ac[j];
                            }
                        } else if constexpr (MODE == GemmMode::kPcF16 ||
                                             MODE == GemmMode::kPgF16) {
                            const float sa = (m < p.M) ? __ldg(p.s_a + m) : 0.0f;
                            bool big = false;
                            if constexpr (MODE == GemmMode::kPcF16) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const int a = (int)ac[j];
                                    big |= (a >= 4194304 || a <= -4194304);
                                }
                            }
                            const bool slow_cvt = __any_sync(0xffffffffu, big);
                            const float* scc = sc + c * 32;
                            uint32_t h2[16];
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                float y0, y1;
                                if constexpr (MODE == GemmMode::kPcF16) {
                                    const float f0 = slow_cvt ? __int2float_rn((int)ac[j])
                                                              : small_int_to_float((int)ac[j]);
                                    const float f1 = slow_cvt ? __int2float_rn((int)ac[j + 1])
                                                              : small_int_to_float((int)ac[j + 1]);
                                    const float2 s2 = *reinterpret_cast<const float2*>(scc + j);
                                    float t0, t1;
                                    fmul2_rn(t0, t1, f0, f1, sa, sa);
                                    fmul2_rn(y0, y1, t0, t1, s2.x, s2.y);
                                } else {
                                    fmul2_rn(y0, y1, __uint_as_float(ac[j]),
                                             __uint_as_float(ac[j + 1]), sa, sa);
                                }
                                h2[j / 2] = pack2_rn(y0, y1, p.out_bf16 != 0);
                            }
                            if (p.tma_store) {
                                if (m_base < p.M && n_c < p.N) {  // warp-uniform
                                    // The staging box is reused: the previous store
                                    // must have read it.
                                    if (store_pending && lane == 0) bulk_wait_group_read0();
                                    __syncwarp();
#pragma unroll
                                    for (int q = 0; q < 4; ++q)
                                        *reinterpret_cast<uint4*>(stage_out + lane * 64 +
                                                                  ((q ^ swz) << 4)) =
                                            make_uint4(h2[4 * q], h2[4 * q + 1], h2[4 * q + 2],
                                                       h2[4 * q + 3]);
                                    fence_proxy_async_smem();
                                    __syncwarp();
                                    if (lane == 0) {
                                        tma_store_2d(&tmap_y, smem_u32(stage_out), n_c, m_base);
                                        bulk_commit_group();
                                    }
                                    store_pending = true;
                                }
                            } else if (m < p.M) {
                                uint16_t* out = static_cast<uint16_t*>(p.out) + (int64_t)m * p.N;
                                const uint16_t* hh = reinterpret_cast<const uint16_t*>(h2);
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (n_c + j < p.N) out[n_c + j] = hh[j];
                            }
                        }
                    }
                }
                if (uses_scales) u_slot = (u_slot + 1 == SD) ? 0 : u_slot + 1;
            }
            first_item = false;
        }
    epi_done:
        cp_async_wait_all();
        if (store_pending && lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Stream-K fix-up: every tile that several CTAs shared gets the sum of their
// int32 partials (exact, any order) and the layer's epilogue, computed as in
// the GEMM epilogue: y = fp16((float(acc) * s_a[m]) * s_w[n]) (or the raw
// int32 sums). One CTA per 32 rows and 64 columns of a tile: lane = row,
// warp w sums the runs of four columns w and w + 8 of its half; rows are
// then written from shared memory, 2 columns per lane.
// ---------------------------------------------------------------------------
struct FixArgs {
    const int32_t* part;
    int part_rows;
    int64_t units;
    int grid;  // CTAs of the GEMM launch
    int num_kb;
    int tiles_m;
    int M, N;
    const float* s_a;
    const float* s_w;
    void* out;
    int out_bf16;
    int raw_s32;
};

constexpr int FIX_THREADS = 256;
constexpr int FIX_STRIDE = 65;  // words per staged row (64 + 1: conflict-free columns)
// Contributors of one tile: at most grid / tiles + 2 CTAs share it.
constexpr int FIX_MAX_CONTRIB = kStreamKMaxCtas + 2;
static_assert(FIX_MAX_CONTRIB <= FIX_THREADS, "one thread per contributor");

__global__ void __launch_bounds__(FIX_THREADS) sk_fixup_kernel(const FixArgs f) {
    __shared__ uint32_t stage[32 * FIX_STRIDE];
    __shared__ const int4* base[FIX_MAX_CONTRIB];  // each contributor's partial tile
    grid_dep_wait();
    grid_dep_launch();
    const int chunks = f.part_rows / 32;
    const int half = blockIdx.x & 1;
    const int tile = (blockIdx.x >> 1) / chunks, chunk = (blockIdx.x >> 1) % chunks;
    const int64_t u0 = (int64_t)tile * f.num_kb;
    const int c_first = sk_cta_of_unit(u0, f.units, f.grid);
    const int c_last = sk_cta_of_unit(u0 + f.num_kb - 1, f.units, f.grid);
    if (c_first == c_last) return;  // one CTA did the whole tile and wrote it
    const int nc = c_last - c_first + 1;
    if ((int)threadIdx.x < nc) {
        // The tile is CTA c's first item (slot 0) exactly when c's run starts
        // inside it, else its last (slot 1).
        const int c = c_first + (int)threadIdx.x;
        const int64_t c_start = (int64_t)c * f.units / f.grid;
        const int slot = (c_start / f.num_kb == tile) ? 0 : 1;
        base[threadIdx.x] =
            reinterpret_cast<const int4*>(f.part) + ((int64_t)c * 2 + slot) * 32 * f.part_rows;
    }
    __syncthreads();
    int tm, tn;
    tile_coords(tile, f.tiles_m, tm, tn);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = chunk * 32 + lane;  // row within the tile
    const int m = tm * BM + r;
    const float sa = (!f.raw_s32 && m < f.M) ? __ldg(f.s_a + m) : 0.0f;
    // All contributors' loads of this thread's two column runs are issued
    // together (contributors outermost, four at a time), so that the sums
    // wait for about one load latency per four contributors.
    int acc[2][4] = {};
#pragma unroll 4
    for (int i = 0; i < nc; ++i) {
        const int4* b = base[i] + r;
        int4 v[2];
#pragma unroll
        for (int pass = 0; pass < 2; ++pass)
            v[pass] = __ldcg(b + (int64_t)(half * 16 + warp + 8 * pass) * f.part_rows);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            acc[pass][0] += v[pass].x;
            acc[pass][1] += v[pass].y;
            acc[pass][2] += v[pass].z;
            acc[pass][3] += v[pass].w;
        }
    }
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int cl = warp + 8 * pass;  // run within the half: columns 4 cl .. 4 cl + 3
        const int a0 = acc[pass][0], a1 = acc[pass][1], a2 = acc[pass][2], a3 = acc[pass][3];
        uint32_t* row = stage + lane * FIX_STRIDE;
        if (f.raw_s32) {
            row[4 * cl] = (uint32_t)a0;
            row[4 * cl + 1] = (uint32_t)a1;
            row[4 * cl + 2] = (uint32_t)a2;
            row[4 * cl + 3] = (uint32_t)a3;
        } else {
            const int n = tn * 128 + half * 64 + 4 * cl;
            const float w0 = (n < f.N) ? __ldg(f.s_w + n) : 0.0f;
            const float w1 = (n + 1 < f.N) ? __ldg(f.s_w + n + 1) : 0.0f;
            const float w2 = (n + 2 < f.N) ? __ldg(f.s_w + n + 2) : 0.0f;
            const float w3 = (n + 3 < f.N) ? __ldg(f.s_w + n + 3) : 0.0f;
            const bool bf16 = f.out_bf16 != 0;
            row[2 * cl] = pack2_rn(__fmul_rn(__fmul_rn(__int2float_rn(a0), sa), w0),
                                   __fmul_rn(__fmul_rn(__int2float_rn(a1), sa), w1), bf16);
            row[2 * cl + 1] = pack2_rn(__fmul_rn(__fmul_rn(__int2float_rn(a2), sa), w2),
                                       __fmul_rn(__fmul_rn(__int2float_rn(a3), sa), w3), bf16);
        }
    }
    __syncthreads();
    // Warp w writes rows w, w + 8, w + 16, w + 24 of the chunk; lane l
    // columns 2 l, 2 l + 1 of the half (int32: 4 l' .. 4 l' + 3 per pass).
    for (int i = warp; i < 32; i += 8) {
        const int mm = tm * BM + chunk * 32 + i;
        if (mm >= f.M) break;
        const uint32_t* row = stage + i * FIX_STRIDE;
        if (f.raw_s32) {
            int32_t* out = static_cast<int32_t*>(f.out) + (int64_t)mm * f.N;
            for (int j = lane; j < 64; j += 32) {
                const int n = tn * 128 + half * 64 + j;
                if (n < f.N) out[n] = (int32_t)row[j];
            }
        } else {
            uint16_t* out = static_cast<uint16_t*>(f.out) + (int64_t)mm * f.N;
            const int n0 = tn * 128 + half * 64 + 2 * lane;
            const uint32_t h01 = row[lane];
            if (n0 + 1 < f.N && (f.N & 1) == 0) {
                *reinterpret_cast<uint32_t*>(out + n0) = h01;
            } else {
                if (n0 < f.N) out[n0] = (uint16_t)(h01 & 0xFFFFu);
                if (n0 + 1 < f.N) out[n0 + 1] = (uint16_t)(h01 >> 16);
            }
        }
    }
}

}  // namespace gemm1

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Row-major 2D tile map: `rows` x `cols` elements of `elem_bytes`, boxes of
// box_rows x box_cols, rows beyond the extent read as zero.
CUresult encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                   const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols, CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <GemmMode MODE, int BSRC, int BN>
cudaError_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                        const gemm1::Params& p, int grid, cudaStream_t stream) {
    using Layout = gemm1::SmemLayout<BSRC, BN, gemm1::tile_groups(MODE, BN)>;
    auto kern = gemm1::gemm_tc1_kernel<MODE, BSRC, BN>;
    // Once per device: the register count the warp-role split assumes, and the
    // shared-memory opt-in.
    static PerDevice<int> attr;
    const cudaError_t e = attr.get([&](int&) {
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != gemm1::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Layout::alloc_bytes);
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, gemm1::NUM_THREADS, Layout::alloc_bytes, stream, ta, tb, ty, p);
}

// Per-channel modes run 128-wide tiles, per-group modes 64-wide ones.
template <int BSRC>
cudaError_t launch_src(GemmMode mode, int bn, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& ty, const gemm1::Params& p, int grid,
                       cudaStream_t stream) {
    switch (mode) {
        case GemmMode::kPcF16:
            return launch_mode<GemmMode::kPcF16, BSRC, 128>(ta, tb, ty, p, grid, stream);
        case GemmMode::kPgF16:
            return bn == 128
                       ? launch_mode<GemmMode::kPgF16, BSRC, 128>(ta, tb, ty, p, grid, stream)
                       : launch_mode<GemmMode::kPgF16, BSRC, 64>(ta, tb, ty, p, grid, stream);
        case GemmMode::kRawS32:
            return launch_mode<GemmMode::kRawS32, BSRC, 128>(ta, tb, ty, p, grid, stream);
        case GemmMode::kRawPgS32:
            return bn == 128
                       ? launch_mode<GemmMode::kRawPgS32, BSRC, 128>(ta, tb, ty, p, grid, stream)
                       : launch_mode<GemmMode::kRawPgS32, BSRC, 64>(ta, tb, ty, p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

CUresult encode_tmap_f16_kmajor(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_cols) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, rows, cols, box_rows,
                     box_cols, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

CUresult encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                            uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, rows, cols, box_rows,
                     box_cols, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

CUresult encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_rows, box_cols,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

CUresult encode_tmap_u8_2d_swizzled(CUtensorMap* map, const void* base, uint64_t rows,
                                    uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                                    CUtensorMapSwizzle swizzle) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, rows, cols, box_rows, box_cols,
                     swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t stream) {
    using namespace gemm1;
    if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.K % 16 != 0) return cudaErrorInvalidValue;
    if (a.M > INT32_MAX / 2 || a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2)
        return cudaErrorInvalidValue;
    const int bsrc = a.b_raw ? a.b_bits : 0;
    if (bsrc != 0 && bsrc != 8 && bsrc != 4) return cudaErrorInvalidValue;
    if (bsrc == 0 && !a.b_img) return cudaErrorInvalidValue;
    if (bsrc == 4 && a.K % 32 != 0) return cudaErrorInvalidValue;
    const bool per_group = (a.mode == GemmMode::kPgF16 || a.mode == GemmMode::kRawPgS32);
    // Tile width: 128 per channel. Per group (whole tiles per CTA): an M128
    // MMA costs the same for N = 64 and N = 128, so 128-wide tiles are taken
    // when they need fewer waves over the SMs (N = 10240: 80 tiles in one
    // wave against 160 in two), else 64-wide ones (less work per tile).
    int BN = 128;
    if (per_group) {
        const int64_t w128 = ((a.N + 127) / 128 * ((a.M + BM - 1) / BM) + num_sms - 1) / num_sms;
        const int64_t w64 = ((a.N + 63) / 64 * ((a.M + BM - 1) / BM) + num_sms - 1) / num_sms;
        BN = (w128 < w64) ? 128 : 64;
    }
    const int kps = stage_kb(bsrc);
    CUtensorMap ta, tb, ty;
    if (encode_tmap_f16_kmajor(&ta, a.a_img, a.M, a.K, BM, BK) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    CUresult rb;
    if (bsrc == 0) {
        rb = encode_tmap_f16_kmajor(&tb, a.b_img, a.N, a.K, BN, BK);
    } else {
        // Raw codes: row n holds K bytes (INT8) or K / 2 bytes (packed INT4);
        // a box is one k-block of BN rows, unswizzled.
        const uint64_t row_bytes = (bsrc == 8) ? (uint64_t)a.K : (uint64_t)a.K / 2;
        rb = encode_tmap_u8_2d(&tb, a.b_raw, a.N, row_bytes, BN, bsrc == 8 ? BK : BK / 2);
    }
    if (rb != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const bool f16_out = (a.mode == GemmMode::kPcF16 || a.mode == GemmMode::kPgF16);
    const bool tma_store =
        f16_out && (a.N % 8 == 0) && (reinterpret_cast<uintptr_t>(a.out) % 16 == 0);
    memset(&ty, 0, sizeof(ty));
    if (tma_store &&
        encode_tmap_f16_2d(&ty, a.out, a.M, a.N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    Params p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.num_blk = (p.K + BK - 1) / BK;
    p.num_kb = (p.num_blk + kps - 1) / kps;
    if (per_group) {
        if (a.group_size <= 0 || a.group_size % BK != 0 || p.K % a.group_size != 0)
            return cudaErrorInvalidValue;
        p.group_kb = a.group_size / BK;
        if (p.group_kb > MAX_SEG_KB) return cudaErrorInvalidValue;  // exact fp32 partials only
        // A segment is tile_groups groups (an even count), a whole number of
        // k-steps.
        const int seg_blk = p.group_kb * tile_groups(a.mode, BN);
        if (seg_blk % kps != 0) return cudaErrorInvalidValue;
        p.seg_kb = seg_blk / kps;
        p.G = p.K / a.group_size;
    } else {
        const int max_seg = MAX_SEG_KB / kps;
        const int nseg = (p.num_kb + max_seg - 1) / max_seg;
        p.seg_kb = (p.num_kb + nseg - 1) / nseg;
        // No group split inside a segment: a stream-K item's segments may be
        // longer than those of a whole tile, never longer than MAX_SEG_KB.
        p.group_kb = MAX_SEG_KB;
        p.G = 1;
    }
    p.num_seg = (p.num_kb + p.seg_kb - 1) / p.seg_kb;
    p.tiles_m = (p.M + BM - 1) / BM;
    p.tiles_n = (p.N + BN - 1) / BN;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.s_wT = per_group ? a.s_wT : nullptr;
    p.out = a.out;
    p.tma_store = tma_store ? 1 : 0;
    p.out_bf16 = a.out_bf16;
    p.timeout_ns = a.timeout_ns;
    p.status = a.status;
    const int tiles = p.tiles_m * p.tiles_n;
    int grid = tiles < num_sms ? tiles : num_sms;
    // Stream-K when whole tiles would leave SMs idle (fewer tiles than SMs,
    // or a last partial wave): every CTA takes an equal run of k-steps.
    // Taken when it shortens the longest CTA's run by at least 12 k-blocks
    // (about the cost of the partial stores and the fix-up launch here:
    // M128 N10240 K2560 went from 32.3 to 28.9 us with 40 against 22).
    const bool per_channel = (a.mode == GemmMode::kPcF16 || a.mode == GemmMode::kRawS32);
    if (per_channel && a.sk_part != nullptr && p.num_kb >= 2) {
        const int64_t units = (int64_t)tiles * p.num_kb;
        int g = num_sms < kStreamKMaxCtas ? num_sms : kStreamKMaxCtas;
        if ((int64_t)g > units) g = (int)units;
        const int64_t dp_kb = (int64_t)((tiles + grid - 1) / grid) * p.num_kb;
        const int64_t sk_kb = (units + g - 1) / g;
        if ((dp_kb - sk_kb) * kps >= 12) {
            p.streamk = 1;
            p.units = units;
            grid = g;
            p.part = a.sk_part;
            p.part_rows = (int)stream_k_part_rows(a.M);
        }
    }
    cudaError_t e;
    if (bsrc == 8)
        e = launch_src<8>(a.mode, BN, ta, tb, ty, p, grid, stream);
    else if (bsrc == 4)
        e = launch_src<4>(a.mode, BN, ta, tb, ty, p, grid, stream);
    else
        e = launch_src<0>(a.mode, BN, ta, tb, ty, p, grid, stream);
    if (e != cudaSuccess || !p.streamk) return e;
    FixArgs f{};
    f.part = p.part;
    f.part_rows = p.part_rows;
    f.units = p.units;
    f.grid = grid;
    f.num_kb = p.num_kb;
    f.tiles_m = p.tiles_m;
    f.M = p.M;
    f.N = p.N;
    f.s_a = p.s_a;
    f.s_w = p.s_w;
    f.out = p.out;
    f.out_bf16 = p.out_bf16;
    f.raw_s32 = (a.mode == GemmMode::kRawS32) ? 1 : 0;
    return launch_pdl(sk_fixup_kernel, tiles * (p.part_rows / 32) * 2, FIX_THREADS, 0, stream, f);
}

}  // namespace cider
