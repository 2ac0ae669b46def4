// chunk_tc.cu -- bf16 chunked prefill on the tcgen05 tensor cores (sm_103a).
//
// Chunked mode of ejkernel kda() ("Algorithm Modes": parallel inside a chunk,
// sequential across chunks) for dk = dv = D in {64, 128}, chunk C = 64.  With the
// chunk-local quantities of the WY / UT-transform form (the representation TileOPs
// DeltaNetChunkFwdOp computes as prepare_wy_repr -> w, u),
//
//   L[t][s] = beta_t (k^_t . k^_s) exp(G_{t-1} - G_s)   (s < t),   T = (I + L)^{-1}
//   P  = T diag(beta),   W = P diag(exp G_{t-1}) K^,   K~_s = exp(G_C - G_s) k^_s
//   Aqk[t][s] = (q~_t . k^_s) exp(G_t - G_s)            (s <= t)
//
// one chunk maps the state S it starts from and its values V to the next state and
// its outputs by a single affine map:
//
//   [ S_next ]   [ exp(G_C) I - K~^T W    K~^T P  ] [ S ]
//   [   O    ] = [ diag(exp G) Q~ - Aqk W  Aqk P   ] [ V ]      =:  E_c [S; V]
//
// (S_next = exp(G_C) S + K~^T U and O = diag(exp G) Q~ S + Aqk U with U = P V - W S.)
// E_c does not depend on the state, so it is built for every chunk in parallel (the
// "prep" role), and a walk over the chunks applies it (the "chain" role):
//
//  * prep -- a group of 256 threads builds E_c for one (sequence, head, chunk) at a
//    time and moves on to the next: TMA loads q, k; tcgen05 products [K;Q] K^T,
//    K^T diag(f) [T'|P], Aqk [T'|P], Z k; a blocked fp32 forward-substitution inverse
//    on CUDA cores; E_c (bf16) goes to scratch by TMA stores.  The next chunk's q, k
//    load is issued as soon as the current chunk has finished reading them.  Two
//    groups share one CTA (and its 512 TMEM columns).
//  * chain -- one CTA per (sequence, head) walks the chunks in order; per chunk one
//    product D^T = [S^T | V^T] E_c^T (M = dv) gives the next state (fp32 in TMEM,
//    stored back as the bf16 operand) and the outputs.  Producer lanes stream E_c and
//    V_c by TMA; an MMA warp issues; eight warps turn the next state into the next
//    operand, four others store o.
//
// Both roles run in one cooperative launch.  The first nch <= SMs/4 CTAs are chains; chain
// i walks the (sequence, head) tasks i, i + nch, i + 2 nch, ... (packed sequences sorted
// longest first), one round of nch tasks after another.  The other CTAs hold the prep
// groups, which take the chunks in (column, chain) order -- column = the chunk's position
// in its chain's walk -- so that every chain's next chunks are built first.  E_c goes
// into a ring of kRing slots per chain: the prep publishes a slot by a release store of
// the chunk's column + 1 to the slot's flag, the chain acquires it before its TMA load and,
// once the load has landed, releases its own "consumed" counter; a prep group waits for
// that counter before it overwrites a slot, so it never runs more than kRing chunks ahead
// of its chain.  The scratch is thus a few MB whatever the sequence length, and E_c lives
// and dies in L2.
//
// Every wait (mbarrier or flag) is bounded; on time-out the kernel records
// KDA_ERR_DEVICE_TIMEOUT in the workspace header and unwinds (no trap).
#include <algorithm>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kC = 64;                        // chunk length
constexpr uint64_t kWaitNs = 2000000000ull;   // bounded waits: 2 s
constexpr int kStatusDeviceTimeout = 8;       // KDA_ERR_DEVICE_TIMEOUT

// E_c slots per chain: the prep's working front spans (prep groups / chains) columns (7.5
// for 32 chains on a 152-SM part), which the ring must hold with room to spare
constexpr int kRing = 16;
constexpr int kMaxChains = 40;                // chain CTAs at most
constexpr int kCounterStride = 32;            // a chain's ring counter (and the item counter) each own a 128-byte line

struct TcParams {
    int nseq, H, T;            // T: equal-length sequence length (unused for varlen)
    int use_l2;
    float scale;
    const int *cu_seqlens;     // nullptr: equal length
    const int *order;          // varlen: sequence indices by decreasing length [nseq] (device)
    const int *round_base;     // varlen: [rounds + 1] first column of each round (device)
    int nc_equal;              // equal length: chunks per sequence (= columns per round)
    const float *beta, *decay; // [rows, H]
    const float *gk;           // per-key-channel decay [rows, H, D] (per-channel kernels) or nullptr
    int decayed_read;          // the delta term reads the decayed state
    const float *A_log;        // [H] or nullptr: decay / gk hold the raw gate (gate_decay)
    const float *dt_bias;      // [H] (scalar decay) or [H, D] (per channel) or nullptr
    int beta_sig, neg_eig;     // beta holds logits: sigmoid, or 2 sigmoid
    int G;                     // value heads per q/k head: H counts value heads, q/k have H / G
    int v_first;               // states value-major [.., D(v), D(k)]
    const float *h0;           // [nseq, H, D, D] or nullptr
    float *hT;                 // [nseq, H, D, D] or nullptr
    const __nv_bfloat16 *q, *k;   // [rows, H, D]
    long rows;                 // token rows of q, k, v
    __nv_bfloat16 *o;          // [rows, H, D]
    __nv_bfloat16 *E;          // scratch: the rings, [nch * ring][D + 64][D + 64]
    uint32_t *flags;           // [nch * ring]: column + 1 of the E_c a slot holds
    int ring;                  // E_c slots per chain (kRing; every column's own slot when the
                               // maps are kept for the backward)
    __nv_bfloat16 *states;     // or nullptr: the state at every chunk start [nseq, H, nc, D, D], bf16
                               // (the walk's own operand precision)
                               // (the reverse walk: the incoming state gradient of every chunk)
    float *dv_out;             // the reverse walk: fp32 value gradient [rows, H, D]
    uint32_t *consumed;        // [nch]: chain i has loaded every E_c of a column below this
    uint32_t *next_item;       // prep items are claimed in order from this counter
    WsHeader *ws;
    int ntask;                 // (sequence, head) tasks
    int nch;                   // chain CTAs (the first ones)
    int rounds;                // ceil(ntask / nch)
};
__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void record_error(WsHeader *ws, int where) {
    if (ws && atomicCAS(&ws->error, 0, kStatusDeviceTimeout) == 0) ws->where = where;
}

// Wait until another CTA has released *f with a value of at least `want` (gpu-scope
// acquire), giving up after limit_ns; on success the async proxy is ordered after the
// acquire (for a TMA load of the data the flag publishes).
__device__ __forceinline__ bool wait_flag_acquire(const uint32_t *f, uint32_t want, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(f) < want) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(64);
    }
    fence_proxy_async_global();
    return true;
}

__device__ __forceinline__ void seq_info(const TcParams &p, int n, long &start, int &len) {
    if (p.cu_seqlens) {
        start = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
    } else {
        start = (long)n * p.T;
        len = p.T;
    }
}
// First column of round r (the chain walk's position where its r-th task begins); r may
// be p.rounds (the total).
__device__ __forceinline__ int round_start(const TcParams &p, int r) {
    return p.cu_seqlens ? p.round_base[r] : r * p.nc_equal;
}
// Task -> (sequence, head): tasks run over the sequences in the order table (longest
// first) and, within a sequence, over its heads.
__device__ __forceinline__ void task_info(const TcParams &p, int task, int &n, int &h) {
    const int rank = task / p.H;
    h = task - rank * p.H;
    n = p.order ? p.order[rank] : rank;
}

// One prep work item: chunk c of sequence n, head h.
struct ChunkItem {
    long row0;         // first token row
    int slot;          // E_c ring slot (= flag index)
    int col;           // column: the chunk's position in its chain's walk
    int chain;         // the chain that consumes it
    int h, nv;         // head; valid tokens in the chunk (1..64)
};

struct PrepCtrl {
    uint64_t bar_mma;
    int fail;
    float gate[2];   // A_log and dt_bias of the chunk's head (raw-gate decay), loaded with beta
    ChunkItem nxi;   // the group's next item, claimed and decoded by one thread while the
    int more;        // current one runs (more = 0: none left)
};
static_assert(sizeof(PrepCtrl) <= 64, "the control block's room in the group's shared memory");

// Prep work items in (column, chain) order: item = column * nch + chain.  Returns false
// for an item past its task's last chunk or past the last task.
__device__ __forceinline__ bool item_info(const TcParams &p, long item, ChunkItem &it) {
    // item < columns x nch < 2^31 (checked on the host), so 32-bit division is exact
    const unsigned u = (unsigned)item;
    const int col = (int)(u / (unsigned)p.nch), chain = (int)(u % (unsigned)p.nch);
    int r;
    if (p.cu_seqlens) {
        int lo = 0, hi = p.rounds;   // round_base[lo] <= col < round_base[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.round_base[mid] <= col) lo = mid; else hi = mid;
        }
        r = lo;
    } else {
        r = col / p.nc_equal;
    }
    const int task = r * p.nch + chain;
    if (task >= p.ntask) return false;
    const int c = col - round_start(p, r);
    int n;
    task_info(p, task, n, it.h);
    long start;
    int len;
    seq_info(p, n, start, len);
    if ((long)c * kC >= len) return false;
    it.row0 = start + (long)c * kC;
    it.nv = min(kC, len - c * kC);
    it.col = col;
    it.chain = chain;
    it.slot = chain * p.ring + col % p.ring;
    return true;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// acc += a * b on a pair of floats by one paired fp32 FMA (each lane rounded as fmaf)
__device__ __forceinline__ void fma2(float2 &acc, float2 a, float2 b) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\tmov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(acc.x), "+f"(acc.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
}

// Named barrier among `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// B = [T' | P] and Bf = diag(f) B (bf16, MN-major SW128: row t, 64 columns s per half,
// half 0 T' = T diag(w), half 1 P = T diag(beta)) for W consecutive columns s.. of row t
// of T.  W = 4, 2, 1: 8-, 4- or 2-byte stores inside one 16-byte chunk.  With PO ("P only")
// just P = T diag(beta) is written, as one 8 KB tile at b.
struct BTiles {
    uint8_t *b, *bf;             // B, Bf: two 8 KB halves each
    const float *w, *beta, *f;   // column weights of T', of P; row weights of Bf
};

template <int W, bool PO = false>
__device__ __forceinline__ void put_b(const BTiles &bt, int t, int s, const float *val) {
    const int off = t * 128 + ((((s >> 3) ^ t) & 7) << 4) + (s & 7) * 2;
    if constexpr (PO) {
        float b1[W];
#pragma unroll
        for (int e = 0; e < W; ++e) b1[e] = val[e] * bt.beta[s + e];
        if constexpr (W == 4)
            *reinterpret_cast<uint2 *>(bt.b + off) = make_uint2(pack_bf16(b1[0], b1[1]), pack_bf16(b1[2], b1[3]));
        else if constexpr (W == 2)
            *reinterpret_cast<uint32_t *>(bt.b + off) = pack_bf16(b1[0], b1[1]);
        else
            *reinterpret_cast<__nv_bfloat16 *>(bt.b + off) = __float2bfloat16_rn(b1[0]);
        return;
    }
    const float ft = bt.f[t];
    float b0[W], b1[W];
#pragma unroll
    for (int e = 0; e < W; ++e) {
        b0[e] = val[e] * bt.w[s + e];
        b1[e] = val[e] * bt.beta[s + e];
    }
    if constexpr (W == 4) {
        *reinterpret_cast<uint2 *>(bt.b + off) = make_uint2(pack_bf16(b0[0], b0[1]), pack_bf16(b0[2], b0[3]));
        *reinterpret_cast<uint2 *>(bt.b + 8192 + off) = make_uint2(pack_bf16(b1[0], b1[1]), pack_bf16(b1[2], b1[3]));
        *reinterpret_cast<uint2 *>(bt.bf + off) =
            make_uint2(pack_bf16(b0[0] * ft, b0[1] * ft), pack_bf16(b0[2] * ft, b0[3] * ft));
        *reinterpret_cast<uint2 *>(bt.bf + 8192 + off) =
            make_uint2(pack_bf16(b1[0] * ft, b1[1] * ft), pack_bf16(b1[2] * ft, b1[3] * ft));
    } else if constexpr (W == 2) {
        *reinterpret_cast<uint32_t *>(bt.b + off) = pack_bf16(b0[0], b0[1]);
        *reinterpret_cast<uint32_t *>(bt.b + 8192 + off) = pack_bf16(b1[0], b1[1]);
        *reinterpret_cast<uint32_t *>(bt.bf + off) = pack_bf16(b0[0] * ft, b0[1] * ft);
        *reinterpret_cast<uint32_t *>(bt.bf + 8192 + off) = pack_bf16(b1[0] * ft, b1[1] * ft);
    } else {
        *reinterpret_cast<__nv_bfloat16 *>(bt.b + off) = __float2bfloat16_rn(b0[0]);
        *reinterpret_cast<__nv_bfloat16 *>(bt.b + 8192 + off) = __float2bfloat16_rn(b1[0]);
        *reinterpret_cast<__nv_bfloat16 *>(bt.bf + off) = __float2bfloat16_rn(b0[0] * ft);
        *reinterpret_cast<__nv_bfloat16 *>(bt.bf + 8192 + off) = __float2bfloat16_rn(b1[0] * ft);
    }
}

// ---------------------------------------------------------------------------------
// T = (I + L)^{-1} for a 64 x 64 strictly-lower L, fp32 in shared memory (row pitch
// kLP = 68 floats: 16-byte aligned rows, and conflict-free A-fragment loads), by the
// NT = 256 threads of one group (named barrier `bar`), on the 4 x 4 grid of 16 x 16 blocks
// (the 2 x 2 block form of the inverse of a lower-triangular matrix, applied twice):
//  * with A = rows/columns 0..31 and B = 32..63: the diagonal blocks T_AA, T_BB, one warp
//    each, by the same form one level down: their 16 x 16 diagonal pieces by forward
//    substitution (half a warp each, one lane per column, the column in registers, each row
//    of L read with 16-byte loads), the piece below by two 16 x 16 products;
//  * T_BA = -T_BB (L_BA T_AA), the 32 x 32 products split into 16 x 8 tiles, one per warp.
// The off-diagonal products run on the tensor cores as warp-level tf32 MMAs (m16n8k8,
// fp32 accumulation; operands rounded to tf32, which keeps 10 fraction bits -- T goes on
// to the bf16 operands B = [T' | P] with 7).  Intermediate products sit in the unused
// upper block of L.  Every block of T is written into B and Bf as soon as it is known.
// ---------------------------------------------------------------------------------
constexpr int kLP = 68;

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// d += a b, m16n8k8, tf32 operands, fp32 accumulators
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// Fragments of row-major fp32 matrices (pitch kLP) at M: the 16 x 8 A tile at rows 0..15,
// columns k0..k0+7, and the 8 x 8 B tile at rows k0..k0+7, columns n0..n0+7 (lane = 4 g + t4).
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const float *M, int k0, int g, int t4) {
    a[0] = to_tf32(M[g * kLP + k0 + t4]);
    a[1] = to_tf32(M[(g + 8) * kLP + k0 + t4]);
    a[2] = to_tf32(M[g * kLP + k0 + t4 + 4]);
    a[3] = to_tf32(M[(g + 8) * kLP + k0 + t4 + 4]);
}
__device__ __forceinline__ void frag_b(uint32_t (&b)[2], const float *M, int k0, int n0, int g, int t4) {
    b[0] = to_tf32(M[(k0 + t4) * kLP + n0 + g]);
    b[1] = to_tf32(M[(k0 + t4 + 4) * kLP + n0 + g]);
}
// A 16 x 8 accumulator tile (rows g, g + 8; columns 2 t4, 2 t4 + 1) stored at M[r][c]
__device__ __forceinline__ void store_c(float *M, const float (&d)[4], int n0, int g, int t4, float sgn) {
    *reinterpret_cast<float2 *>(M + g * kLP + n0 + 2 * t4) = make_float2(sgn * d[0], sgn * d[1]);
    *reinterpret_cast<float2 *>(M + (g + 8) * kLP + n0 + 2 * t4) = make_float2(sgn * d[2], sgn * d[3]);
}

template <int NT, bool PO = false, typename IdleWork>
__device__ void invert_unit_lower_64(float *sL, float *sT, const BTiles &bt, int tid, int bar,
                                     IdleWork &&idle) {
    static_assert(NT == 256, "the work split below assumes 256 threads");
    constexpr int P = kLP;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    if (warp < 2) {
        // diagonal 32 x 32 block `warp` (T_AA, T_BB) in 16 x 16 pieces: lanes 0-15 take the
        // columns of its first diagonal piece, lanes 16-31 those of its second, each by
        // forward substitution with the column in registers,
        //   x_r = delta_rj - sum_{s<r} L[r][s] x_s,
        // the row of L read by 16-byte loads (the terms with earlier x_s are summed while the
        // later ones are still being computed); then the piece below the diagonal,
        // T_10 = -T_11 (L_10 T_00), by two warp-level tf32 MMA steps, L_10 T_00 kept in L's
        // unused upper piece of the block
        const int b0 = 32 * warp, j = lane & 15;
        const int o = b0 + 16 * (lane >> 4);   // first row and column of this lane's piece
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float4 *Lr = reinterpret_cast<const float4 *>(sL + (o + r) * P + o);
            float2 acc = make_float2(0.f, 0.f);   // sum_{s<r} L[r][s] x_s, by pairs of s
#pragma unroll
            for (int m4 = 0; m4 < (r + 3) / 4; ++m4) {
                const float4 v = Lr[m4];
                const int s0 = 4 * m4;
                if (s0 + 1 < r) fma2(acc, make_float2(v.x, v.y), make_float2(x[s0], x[s0 + 1]));
                else if (s0 < r) acc.x = fmaf(v.x, x[s0], acc.x);
                if (s0 + 3 < r) fma2(acc, make_float2(v.z, v.w), make_float2(x[s0 + 2], x[s0 + 3]));
                else if (s0 + 2 < r) acc.x = fmaf(v.z, x[s0 + 2], acc.x);
            }
            x[r] = ((r == j) ? 1.f : 0.f) - (acc.x + acc.y);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(o + r) * P + o + j] = x[r];
        if (lane < 16)   // T_01 = 0
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(b0 + r) * P + b0 + 16 + j] = 0.f;
        __syncwarp();
        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {   // L_10 T_00
                uint32_t a[4], b[2];
                frag_a(a, sL + (b0 + 16) * P + b0, k0, g, t4);
                frag_b(b, sT + b0 * P + b0, k0, 8 * nt, g, t4);
                mma_tf32(y[nt], a, b);
            }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) store_c(sL + b0 * P + b0 + 16, y[nt], 8 * nt, g, t4, 1.f);
        __syncwarp();
        float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int k0 = 0; k0 < 16; k0 += 8) {   // T_11 (L_10 T_00)
                uint32_t a[4], b[2];
                frag_a(a, sT + (b0 + 16) * P + b0 + 16, k0, g, t4);
                frag_b(b, sL + b0 * P + b0 + 16, k0, 8 * nt, g, t4);
                mma_tf32(z[nt], a, b);
            }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) store_c(sT + (b0 + 16) * P + b0, z[nt], 8 * nt, g, t4, -1.f);
    } else {
        // the other 192 threads zero the four 16 x 16 blocks of B and Bf above the diagonal
        // 32 x 32 blocks: 4 blocks x 16 rows x 2 chunks x 4 tiles (B, Bf; T' and P halves),
        // or of P alone
        const int zt = tid - 64;
        for (int idx = zt; idx < 4 * 16 * 2 * (PO ? 1 : 4); idx += NT - 64) {
            const int ch = idx & 1, r = (idx >> 1) & 15, blk = (idx >> 5) & 3, tile = idx >> 7;
            const int bi = blk >> 1, bj = 2 + (blk & 1);           // (0,2) (0,3) (1,2) (1,3)
            const int t = 16 * bi + r;
            uint8_t *base = (tile & 1 ? bt.bf : bt.b) + (tile >> 1) * 8192;
            *reinterpret_cast<uint4 *>(base + t * 128 + ((((2 * bj + ch) ^ t) & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        idle();   // work of the caller's that fits in the substitution's shadow
    }
    named_sync(bar, NT);
    // X2 = L_BA T_AA (rows 32..63, columns 0..31) into L's free upper-right 32 x 32 block;
    // T_AA[0:16][16:32] = 0, so the right half of X2 sums over k >= 16 only
    const int mi = warp >> 2, ni = warp & 3;
    float *X2 = sL + 32;
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8) {
            if (ni >= 2 && k0 < 16) continue;
            uint32_t a[4], b[2];
            frag_a(a, sL + (32 + 16 * mi) * P, k0, g, t4);
            frag_b(b, sT, k0, 8 * ni, g, t4);
            mma_tf32(d, a, b);
        }
        store_c(X2 + 16 * mi * P, d, 8 * ni, g, t4, 1.f);
    }
    // the diagonal blocks into B and Bf: 2 blocks x 32 rows x 8 quads of columns (the
    // quads above a row's diagonal are zeros written by the substitution)
    for (int w = tid; w < 512; w += NT) {
        const int blk = w >> 8, r = (w >> 3) & 31, c4 = (w & 7) * 4;
        const float4 d = *reinterpret_cast<const float4 *>(sT + (32 * blk + r) * P + 32 * blk + c4);
        const float dv[4] = {d.x, d.y, d.z, d.w};
        put_b<4, PO>(bt, 32 * blk + r, 32 * blk + c4, dv);
    }
    named_sync(bar, NT);
    // T_BA = -T_BB X2; T_BB[0:16][16:32] = 0, so rows 32..47 sum over k < 16 only
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 8) {
            if (mi == 0 && k0 >= 16) continue;
            uint32_t a[4], b[2];
            frag_a(a, sT + (32 + 16 * mi) * P + 32, k0, g, t4);
            frag_b(b, X2, k0, 8 * ni, g, t4);
            mma_tf32(d, a, b);
        }
        const float v0[2] = {-d[0], -d[1]}, v1[2] = {-d[2], -d[3]};
        put_b<2, PO>(bt, 32 + 16 * mi + g, 8 * ni + 2 * t4, v0);
        put_b<2, PO>(bt, 32 + 16 * mi + g + 8, 8 * ni + 2 * t4, v1);
    }
    fence_proxy_async();   // B, Bf are tensor-core operands
    tc_fence_before();
    named_sync(bar, NT);
}

// 8 fp32 -> one 16-byte group of bf16
__device__ __forceinline__ uint4 pack8(const float *f) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                      pack_bf16(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack8un(const uint32_t *u) {   // of the negated values
    return make_uint4(pack_bf16(-__uint_as_float(u[0]), -__uint_as_float(u[1])),
                      pack_bf16(-__uint_as_float(u[2]), -__uint_as_float(u[3])),
                      pack_bf16(-__uint_as_float(u[4]), -__uint_as_float(u[5])),
                      pack_bf16(-__uint_as_float(u[6]), -__uint_as_float(u[7])));
}
__device__ __forceinline__ uint4 pack8u(const uint32_t *u) {
    return make_uint4(pack_bf16(__uint_as_float(u[0]), __uint_as_float(u[1])),
                      pack_bf16(__uint_as_float(u[2]), __uint_as_float(u[3])),
                      pack_bf16(__uint_as_float(u[4]), __uint_as_float(u[5])),
                      pack_bf16(__uint_as_float(u[6]), __uint_as_float(u[7])));
}

// ---------------------------------------------------------------------------------
// prep -- one group of 256 threads builds E_c chunk after chunk.  The two warps w and
// w + 4 of a group share TMEM lane quadrant w % 4 and split each result row's columns
// between them.  Rows of an M = 128 result: 32 q + lane; of an M = 64 result:
// 16 q + lane for lane < 16.
// ---------------------------------------------------------------------------------
constexpr int kGroupThreads = 256;
constexpr int kTcThreads = 512;               // prep: two groups; chain: 14 warps used
// The group's thread that issues the E_c stores, waits for them and publishes E_c: a thread
// other than the MMA issuer (whose release would also wait for its MMAs), in warp 4, which
// issues no loads that the release would have to wait for.
constexpr int kStoreThread = 128;

template <int D>
struct PrepSmem {
    static constexpr int NB = D / 64;
    static constexpr int KQ = 0;                      // [K;Q] tile, K-major SW128: NB x 16 KB
    static constexpr int R1 = KQ + NB * 16384;        // L, T fp32 [64][kLP]; later Z1, Z2
    static constexpr int R2 = R1 + 35840;             // Bf, B: MN-major [64 t][128], 16 KB each
    static constexpr int R3 = R2 + 32768;             // Aqk: K-major [64 t][64 s], 8 KB
    static constexpr int MISC = R3 + 8192;            // per-token scalars, 10 x 64 floats
    static constexpr int CTRL = MISC + 10 * 64 * 4;   // the group's mbarriers and status
    static constexpr int GROUP = ((CTRL + 64 + 1023) / 1024) * 1024;   // one group's share
};

struct ChunkItem;
struct PrepCtrl;

__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// q or k of one chunk into its rows of the [K;Q] region (K-major SW128; k rows 0-63, q rows
// 64-127 of each 64-column block) by 16-byte cp.async copies spread over the group's warps
// other than 0 (the MMA issuer) and 4 (the store thread, whose flag release would wait for
// loads in flight).  These go through the load path, not the TMA unit, where they would
// queue behind the E_c stores.  Rows past the token array are filled with zeros.
template <int D, bool OPT>
__device__ __forceinline__ void load_rows(const TcParams &p, uint8_t *sKQ, const ChunkItem &it,
                                          int tid, bool q) {
    constexpr int PPR = D / 8;                               // 16-byte pieces per row
    const __nv_bfloat16 *g = q ? p.q : p.k;
    const int w = tid >> 5;
    if (w == 0 || w == 4) return;
    const int lt = (w < 4 ? tid - 32 : tid - 64);   // 0 .. 191
    for (int pidx = lt; pidx < 64 * PPR; pidx += kGroupThreads - 64) {
        const int row = pidx / PPR, pc = pidx % PPR;
        const long grow = it.row0 + row;
        const bool in = grow < p.rows;
        const int G = OPT ? p.G : 1;   // value heads per q/k head
        const __nv_bfloat16 *src = g + ((in ? grow : 0) * (p.H / G) + it.h / G) * D + 8 * pc;
        uint8_t *dst = sKQ + (pc >> 3) * 16384 + (q ? 8192 : 0) + row * 128 + (((pc & 7) ^ (row & 7)) << 4);
        cp_async16(dst, src, in ? 16u : 0u);
    }
    cp_async_commit();
}
// beta, decay of one chunk into the per-token scalars (zero past the chunk's valid tokens;
// decay zero when absent); with a raw-gate decay also A_log and dt_bias of the head, so that
// no global load sits on the prefix's path
template <bool OPT>
__device__ __forceinline__ void load_scalars(const TcParams &p, float *mbeta, float *mdec, float *gate,
                                             const ChunkItem &it, int tid) {
    const int t = tid - 64;   // warps 2, 3
    if (t >= 0 && t < 64) {
        const long gi = (it.row0 + (t < it.nv ? t : 0)) * p.H + it.h;
        cp_async4(mbeta + t, p.beta + gi, t < it.nv ? 4u : 0u);
        cp_async4(mdec + t, p.decay ? p.decay + gi : p.beta + gi, (t < it.nv && p.decay) ? 4u : 0u);
        if (OPT && p.A_log && t < 2) {
            const float *src = t == 0 ? p.A_log + it.h : (p.dt_bias ? p.dt_bias + it.h : p.A_log);
            cp_async4(gate + t, src, (t == 0 || p.dt_bias) ? 4u : 0u);
        }
    }
    cp_async_commit();
}

// E_c of column `col` is in global memory in `slot` (its bulk stores have completed):
// release the slot's flag
__device__ __forceinline__ void release_slot(const TcParams &p, int slot, int col) {
    fence_proxy_async_global();
    st_release_gpu(p.flags + slot, (uint32_t)col + 1u);
}

// Before E_c of column `col` goes into its chain's ring: wait until the chain has loaded
// the E_c that the slot held (column col - kRing), giving up after limit_ns; the async
// proxy is then ordered after the acquire (the slot is written by TMA stores).
// seen: the group's record of the counters it has read (shared memory, one per chain): a
// counter already seen at or past `need` is not read again -- that earlier acquire orders the
// slot's reuse just as well -- so the common case costs no round trip to the counter's line,
// which may sit in the other die's L2.
__device__ __forceinline__ bool wait_slot_free(const TcParams &p, int chain, int col, uint64_t limit_ns,
                                               uint32_t *seen) {
    if (col >= p.ring) {
        const uint32_t need = (uint32_t)(col - p.ring + 1);
        if (seen[chain] < need) {
            // a group that has run a full ring ahead waits for its chain: the wait backs off
            // (64 ns to 1 us), so that many waiting groups do not crowd the counter's line
            // while the chain's release has to land on it
            const uint64_t t0 = globaltimer_ns();
            uint32_t v, ns = 64;
            while ((v = ld_acquire_gpu(p.consumed + chain * kCounterStride)) < need) {
                if (globaltimer_ns() - t0 > limit_ns) return false;
                __nanosleep(ns);
                ns = ns < 1024 ? 2 * ns : 1024;
            }
            seen[chain] = v;
        }
    }
    fence_proxy_async_global();
    return true;
}

// Prep work items: columns x chains
__device__ __forceinline__ long prep_items(const TcParams &p) {
    return (long)round_start(p, p.rounds) * p.nch;
}

// The next prep item, in (column, chain) order, from the launch's shared counter: a group
// that finishes early takes the next chunk, so the prep's front stays as narrow as the
// work allows (no group holds a chunk far ahead of the others while its chain waits for
// another).  Items past a task's last chunk are skipped.  The item is decoded into `it`
// (shared memory) by the claiming thread, so the decode (a few integer divisions, ~1.7 K
// cycles with their loads) runs in its shadow instead of on every thread's path.  Returns 0
// when no item is left.
__device__ __forceinline__ int claim_item(const TcParams &p, long n_items, ChunkItem &it) {
    while (true) {
        const long x = (long)atomicAdd(p.next_item, 1u);
        if (x >= n_items) return 0;
        ChunkItem t;
        if (item_info(p, x, t)) {
            it = t;
            return 1;
        }
    }
}

// The two prep groups of a CTA run the same phases; when they run them at the same time
// they contend for issue slots and shared memory.  With `stagger`, group 1 starts its first
// chunk only when group 0 has finished its first epilogue 1 (named barrier kStaggerBar:
// group 0 arrives once, group 1 waits once); the offset of about a third of a chunk
// persists (measured: 0.962 -> 0.949 ms on a 32 x 32768-token prefill; a two-thirds offset
// gained nothing).
constexpr int kStaggerBar = 3;
// Group g's warps 0-2 meet at named barrier g + kGateBarOffset (4, 5) when the decay comes
// from a raw gate: warps 1 and 2 transform it, warp 0 then takes the prefix.
constexpr int kGateBarOffset = 3;

// OPT: the kda_options code paths (decayed read, gate and beta prologues, grouped heads);
// the plain instantiation compiles them out.
template <int D, bool OPT>
__device__ __forceinline__ void prep_group(const CUtensorMap *map_q, const CUtensorMap *map_k,
                                           const CUtensorMap *map_E, const TcParams &p,
                                           uint8_t *sm, uint32_t tm, int tid, int bar, bool stagger) {
    using Ly = PrepSmem<D>;
    constexpr int NB = D / 64;
    constexpr int R = D + 64;
    PrepCtrl *ctl = reinterpret_cast<PrepCtrl *>(sm + Ly::CTRL);
    __shared__ uint32_t s_seen[2][kMaxChains];   // per group: the ring counters last read
    uint32_t *seen = s_seen[bar - 1];
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hh = warp >> 2;
    if (tid < kMaxChains) seen[tid] = 0;   // (first read after the loop's barriers)
    const int i128 = 32 * q4 + lane;
    const int i64 = 16 * q4 + lane;
    const bool has64 = lane < 16;
    const uint32_t tq = (uint32_t)(32 * q4) << 16;   // this warp's TMEM lane quadrant

    uint8_t *sKQ = sm + Ly::KQ;
    float *sL = reinterpret_cast<float *>(sm + Ly::R1);
    float *sT = sL + 64 * kLP;
    uint8_t *sZ1 = sm + Ly::R1;
    // Z2 and, 8 KB after it, the diagonal block of MMA3b's A operand: clear of the V-column
    // staging block of E_c (R1 + R*128 .. + R*128 at D = 64), which epilogue 2 writes too
    uint8_t *sZ2 = sm + Ly::R1 + (D == 128 ? D * 128 : 32768);
    static_assert(D == 128 ? (D * 128 + 16384 <= NB * (R * 128)) : (32768 >= (NB + 1) * (R * 128)),
                  "MMA3b's A operand overlaps the V-column staging");
    uint8_t *sBf = sm + Ly::R2;
    uint8_t *sB = sm + Ly::R2 + 16384;
    uint8_t *sA = sm + Ly::R3;
    // E_c staging (K-major SW128, NB + 1 blocks of R rows): reuses R1..R3 once they are dead
    // (the V-column block NB after MMA2, the state-column blocks after MMA3)
    uint8_t *sEst = sm + Ly::R1;
    static_assert(Ly::R1 + (NB + 1) * (R * 128) <= Ly::MISC, "E_c staging overlaps the scalars");
    float *mbeta = reinterpret_cast<float *>(sm + Ly::MISC);
    float *mdec = mbeta + 64, *mG = mdec + 64, *mGp = mG + 64, *mkn = mGp + 64, *mqn = mkn + 64;
    float *mf = mqn + 64, *meg = mf + 64, *mcw = meg + 64;
    float *mce = mcw + 64;   // column factor exp(G_e - G_s), e the last token of s's 32-token half

    const bool lead = stagger && bar == 1, follow = stagger && bar == 2;
    if (follow) named_sync(kStaggerBar, 2 * kGroupThreads);
    const long n_items = prep_items(p);
    if (tid == 0) ctl->more = claim_item(p, n_items, ctl->nxi);
    named_sync(bar, kGroupThreads);
    if (!ctl->more) {
        if (lead) named_arrive(kStaggerBar, 2 * kGroupThreads);
        return;
    }
    ChunkItem cur = ctl->nxi;
    named_sync(bar, kGroupThreads);   // everyone has read the item before it is claimed again
    load_rows<D, OPT>(p, sKQ, cur, tid, true);
    load_rows<D, OPT>(p, sKQ, cur, tid, false);
    load_scalars<OPT>(p, mbeta, mdec, ctl->gate, cur, tid);
    // store thread: the slot (and column) whose stores are in flight and not yet published,
    // and the one whose state-column blocks wait in the staging area
    int pend = -1, pend_col = 0, staged = -1, staged_col = 0;

    for (uint32_t it = 0;; ++it) {
        const uint32_t ph = it & 1;   // bar_mma completes three times per chunk
        const int nv = cur.nv;
        const bool gated = OPT && p.A_log && p.decay;   // decay holds the raw gate
        cp_async_wait_all();   // this thread's share of q, k, beta, decay ...
        fence_proxy_async();   // ... visible to the tensor core behind the barrier
        named_sync(bar, kGroupThreads);
        bool ok = ctl->fail == 0;
        if (tid == kStoreThread && staged >= 0) {   // the previous chunk's state-column blocks of E_c
            for (int kb = 0; kb < NB; ++kb)
                tma_store_3d(map_E, sEst + kb * (R * 128), kb * 64, 0, staged);
            bulk_commit();
            pend = staged;
            pend_col = staged_col;
            staged = -1;
        }

        // ---- MMA1: D1[0:128, 0:64] = [K; Q] K^T  (contraction over the head dim)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(128, 64, false, false);
            const uint32_t a0 = smem_u32(sKQ);
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16_ss(tm, desc_kmajor_sw128(a0, 128, ks), desc_kmajor_sw128(a0, 128, ks), id,
                            ks > 0 ? 1u : 0u);
            mma_commit(&ctl->bar_mma);
        }
        if (gated && (warp == 1 || warp == 2)) {   // the decay from the raw gate, a token per thread
            const int t = tid - 32;                  // (zero past the valid tokens)
            mdec[t] = t < nv ? gate_decay(mdec[t], ctl->gate[0], ctl->gate[1]) : 0.f;
            named_arrive(bar + kGateBarOffset, 96);
        }
        if (warp == 0) {   // in-chunk cumulative log-decay: lane owns tokens 2 lane, 2 lane + 1
            if (gated) named_sync(bar + kGateBarOffset, 96);
            const float d0 = mdec[2 * lane], d1 = mdec[2 * lane + 1];

            float incl = d0 + d1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const float excl = incl - (d0 + d1);
            mGp[2 * lane] = excl;
            mG[2 * lane] = excl + d0;
            mGp[2 * lane + 1] = excl + d0;
            mG[2 * lane + 1] = incl;
            // G at the last token of each 32-token half: lanes 15 and 31 hold tokens 31, 63
            const float gend = __shfl_sync(0xffffffffu, incl, lane < 16 ? 15 : 31);
            mce[2 * lane] = __expf(gend - (excl + d0));
            mce[2 * lane + 1] = __expf(gend - incl);
        }
        if (OPT && warp == 3 && p.beta_sig) {   // beta from logits (zero past the valid tokens)
            mbeta[2 * lane] = 2 * lane < nv ? beta_of(mbeta[2 * lane], 1, p.neg_eig) : 0.f;
            mbeta[2 * lane + 1] = 2 * lane + 1 < nv ? beta_of(mbeta[2 * lane + 1], 1, p.neg_eig) : 0.f;
        }
        if (tid >= 128 && ok) {   // query norms: two threads per row, each summing half of its chunks
            const int t = (tid - 128) >> 1, part = tid & 1;
            float ss = 0.f;
#pragma unroll
            for (int cc = 0; cc < NB * 4; ++cc) {
                // logical chunk `chunk` sits at (chunk ^ t) % 8 in its block; reading that slot
                // keeps the eight rows of a warp on eight different bank groups
                const int chunk = part * NB * 4 + cc;
                const uint4 w = *reinterpret_cast<const uint4 *>(sKQ + (chunk >> 3) * 16384 + 8192 +
                                                                 t * 128 + (((chunk ^ t) & 7) << 4));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = bf16lo(ws[e]), b = bf16hi(ws[e]);
                    ss = fmaf(a, a, fmaf(b, b, ss));
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (part == 0) mqn[t] = p.use_l2 ? p.scale / fmaxf(sqrtf(ss), kNormEps) : p.scale;
        }
        named_sync(bar, kGroupThreads);   // the log-decay prefix is in place
        if (tid < 64) meg[tid] = __expf(mG[tid]);
        if (ok && !mbar_wait(&ctl->bar_mma, ph, kWaitNs)) ctl->fail = 1;
        tc_fence_after();

        // ---- epilogue 1: norms, L (fp32, smem) and Aqk (bf16 operand); columns 32 hh ..
        {
            uint32_t r[32];
            tmem_ld32(tm + tq + 32 * hh, r);
            tmem_ld_wait();
            if (i128 < 64 && (i128 >> 5) == hh) {   // this half holds the Gram diagonal of row i128
                float diag = 0.f;
#pragma unroll
                for (int s = 0; s < 32; ++s)
                    if (s == (i128 & 31)) diag = __uint_as_float(r[s]);
                mkn[i128] = p.use_l2 ? 1.f / fmaxf(sqrtf(diag), kNormEps) : 1.f;
            }
            // the previous chunk's E_c stores must have read the staging area before
            // it is overwritten behind this barrier
            if (tid == kStoreThread) bulk_wait_read0();
            named_sync(bar, kGroupThreads);
            const float gC = mG[63];
            // Row t's block of 32 tokens against this warp's 32 columns (warp-uniform): above
            // the diagonal all zeros; below it the decay factor exp(R_t - G_s) splits into
            // exp(R_t - G_e) exp(G_e - G_s) with e the last column of the half (both <= 1 for
            // a non-increasing G), a row factor and the column factors mce; on the diagonal
            // block each entry takes its own exponential.
            const bool lrows = i128 < 64;
            const int t = lrows ? i128 : i128 - 64;
            const int cb = t >> 5;
            // R_t: G_{t-1} when the delta term reads h_{t-1}, G_t when it reads the decayed memory
            const float kt = mkn[t], bt = mbeta[t];
            const float gpt = lrows ? ((OPT && p.decayed_read) ? mG[t] : mGp[t]) : mG[t];
            if (lrows && hh == 0) {
                mf[t] = t < nv ? __expf(gC - mG[t]) * kt : 0.f;
                mcw[t] = bt * __expf(gpt) * kt;   // column weight of T' = T diag(beta e^{G_{s-1}} kn)
            }
            // L: beta_t kn_t kn_s k_t.k_s e^{R_t - G_s} (s < t);  Aqk: qn_t kn_s q_t.k_s e^{G_t - G_s} (s <= t)
            const float rbase = t < nv ? (lrows ? bt * kt : mqn[t]) : 0.f;
            float v[32];
            if (cb < hh || rbase == 0.f) {
#pragma unroll
                for (int s2 = 0; s2 < 32; ++s2) v[s2] = 0.f;
            } else if (cb > hh) {
                const float rf = rbase * __expf(gpt - mG[32 * hh + 31]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 a = reinterpret_cast<const float4 *>(mkn + 32 * hh)[e];
                    const float4 c = reinterpret_cast<const float4 *>(mce + 32 * hh)[e];
                    v[4 * e] = rf * a.x * c.x * __uint_as_float(r[4 * e]);
                    v[4 * e + 1] = rf * a.y * c.y * __uint_as_float(r[4 * e + 1]);
                    v[4 * e + 2] = rf * a.z * c.z * __uint_as_float(r[4 * e + 2]);
                    v[4 * e + 3] = rf * a.w * c.w * __uint_as_float(r[4 * e + 3]);
                }
            } else {
                const int lim = lrows ? (t & 31) : (t & 31) + 1;   // columns s2 < lim are kept
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 a = reinterpret_cast<const float4 *>(mkn + 32 * hh)[e];
                    const float4 g = reinterpret_cast<const float4 *>(mG + 32 * hh)[e];
                    const float kn4[4] = {a.x, a.y, a.z, a.w}, g4[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s2 = 4 * e + u;
                        const float val = rbase * kn4[u] * __uint_as_float(r[s2]) * __expf(gpt - g4[u]);
                        v[s2] = s2 < lim ? val : 0.f;
                    }
                }
            }
            if (lrows) {
                float *Lrow = sL + t * kLP + 32 * hh;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    reinterpret_cast<float4 *>(Lrow)[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            } else {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = 4 * hh + cc;
                    *reinterpret_cast<uint4 *>(sA + t * 128 + ((chunk ^ (t & 7)) << 4)) = pack8(v + 8 * cc);
                }
            }
        }
        fence_proxy_async();
        named_sync(bar, kGroupThreads);
        ok = ctl->fail == 0;
        if (lead && it == 0) named_arrive(kStaggerBar, 2 * kGroupThreads);
        // ---- T = (I + L)^{-1}, written as B = [T' | P], Bf = diag(f) B (MN-major: row t, columns s).
        // In the substitution's shadow, one thread of the idle warps claims this group's next
        // chunk (the atomic and the decode off every path) and starts its q and k towards L2,
        // ahead of their load after MMA3; everyone reads the item after the inverse.
        invert_unit_lower_64<kGroupThreads>(sL, sT, BTiles{sB, sBf, mcw, mbeta, mf}, tid, bar, [&] {
            if (tid == 64) {
                ctl->more = claim_item(p, n_items, ctl->nxi);
                if (ctl->more) {
                    const ChunkItem &n = ctl->nxi;
                    const int hq = OPT ? n.h / p.G : n.h;
                    for (int kb = 0; kb < NB; ++kb) {
                        tma_prefetch_l2_3d(map_q, kb * 64, hq, (int)n.row0);
                        tma_prefetch_l2_3d(map_k, kb * 64, hq, (int)n.row0);
                    }
                }
            }
        });
        const bool more = ctl->more != 0;
        const ChunkItem nx = ctl->nxi;


        // ---- MMA2: D2a[:, 0:128] = K^T diag(f) [T'|P]  (M = D);  D2b[:, 128:256] = Aqk [T'|P]
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t ida = idesc_bf16_f32(D, 128, true, true);
            const uint32_t idb = idesc_bf16_f32(64, 128, false, true);
            const uint32_t kq = smem_u32(sKQ), bf = smem_u32(sBf), bb = smem_u32(sB), aa = smem_u32(sA);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm, desc_mnmajor_sw128(kq, 128, ks), desc_mnmajor_sw128(bf, 64, ks), ida,
                            ks > 0 ? 1u : 0u);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm + 128, desc_kmajor_sw128(aa, 64, ks), desc_mnmajor_sw128(bb, 64, ks), idb,
                            ks > 0 ? 1u : 0u);
            mma_commit(&ctl->bar_mma);
        }
        // The previous chunk's E_c is published while MMA2 runs (the whole group waits for it
        // anyway): its stores (this chunk's start, the previous MMA3) have completed, and the
        // gpu-scope release, about a thousand cycles, overlaps the MMA.
        if (tid == kStoreThread && pend >= 0) {
            bulk_wait0();
            release_slot(p, pend, pend_col);
            pend = -1;
        }
        if (ok && !mbar_wait(&ctl->bar_mma, ph ^ 1u, kWaitNs)) ctl->fail = 1;
        tc_fence_after();

        // ---- epilogue 2: Z1, Z2 operands (column half 0); the V columns of E (half 1)
        {
            uint32_t v[64];
            tmem_ld32(tm + tq + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(v));
            tmem_ld32(tm + tq + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            tmem_ld_wait();
            const bool has_row = (D == 128) || has64;
            const int i = (D == 128) ? i128 : i64;
            if (has_row) {
                if (hh == 0) {   // Z1[i][s]: K-major operand, rows i
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        *reinterpret_cast<uint4 *>(sZ1 + i * 128 + ((cc ^ (i & 7)) << 4)) = pack8u(v + 8 * cc);
                } else {         // E[i][D + s] = (K~^T P)[i][s] -> staging block NB
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        *reinterpret_cast<uint4 *>(sEst + NB * (R * 128) + i * 128 + ((cc ^ (i & 7)) << 4)) =
                            pack8u(v + 8 * cc);
                }
            }
            tmem_ld32(tm + tq + 128 + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(v));
            tmem_ld32(tm + tq + 128 + 64 * hh + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            tmem_ld_wait();
            if (has64) {
                const int t = i64;
                if (hh == 0) {   // A of MMA3b: [-Z2 | diag(a)], a_t = exp(G_t) q-scale_t (0 past nv)
                    const float a = t < nv ? meg[t] * mqn[t] : 0.f;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int off = t * 128 + ((cc ^ (t & 7)) << 4);
                        *reinterpret_cast<uint4 *>(sZ2 + off) = pack8un(v + 8 * cc);
                        float dg[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) dg[e] = (8 * cc + e == t) ? a : 0.f;
                        *reinterpret_cast<uint4 *>(sZ2 + 8192 + off) = pack8(dg);
                    }
                } else {         // E[D + t][D + s] = (Aqk P)[t][s] -> staging block NB
                    const int rr = D + t;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        *reinterpret_cast<uint4 *>(sEst + NB * (R * 128) + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
                            pack8u(v + 8 * cc);
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(bar, kGroupThreads);
        ok = ctl->fail == 0;

        // ---- MMA3: D3a[:, 0:D] = Z1 k  (M = D);  D3b[:, 128:128+D] = diag(a) q - Z2 k  (M = 64)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t ida = idesc_bf16_f32(D, D, false, true);
            const uint32_t idb = idesc_bf16_f32(64, D, false, true);
            const uint32_t kq = smem_u32(sKQ), z1 = smem_u32(sZ1), z2 = smem_u32(sZ2);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm, desc_kmajor_sw128(z1, D, ks), desc_mnmajor_sw128(kq, 128, ks), ida,
                            ks > 0 ? 1u : 0u);
            for (int ks = 0; ks < 8; ++ks)   // [-Z2 | diag(a)] [k; q]: the q~ rows of E_c in one go
                mma_bf16_ss(tm + 128, desc_kmajor_sw128(z2, 64, ks), desc_mnmajor_sw128(kq, 128, ks),
                            idb, ks > 0 ? 1u : 0u);
            mma_commit(&ctl->bar_mma);
        }
        if (tid == kStoreThread && ok) {   // the V-column block, to drain during MMA3 and epilogue 3
            if (wait_slot_free(p, cur.chain, cur.col, kWaitNs, seen)) {   // the ring slot has been read
                tma_store_3d(map_E, sEst + NB * (R * 128), NB * 64, 0, cur.slot);
                bulk_commit();
            } else {
                ctl->fail = 1;
                record_error(p.ws, 3);
            }
        }
        if (ok && !mbar_wait(&ctl->bar_mma, ph, kWaitNs)) ctl->fail = 1;
        tc_fence_after();
        // [K;Q] is free once MMA3 has read it, beta and decay after the inverse: the next
        // chunk's load starts now
        if (ok && more) {
            load_rows<D, OPT>(p, sKQ, nx, tid, true);
            load_rows<D, OPT>(p, sKQ, nx, tid, false);
            load_scalars<OPT>(p, mbeta, mdec, ctl->gate, nx, tid);
        }

        // ---- epilogue 3: the state columns of E; column half hh covers [hh D/2, (hh+1) D/2)
        {
            constexpr int HALF = D / 2;
            const float gamma_c = meg[63];
            const bool has_row = (D == 128) || has64;
            const int i = (D == 128) ? i128 : i64;
            const int t = i64;   // E[D + t][j] = exp(G_t) q~_t[j] - (Aqk W)[t][j] = D3b[t][j]
            static_assert(HALF == 64 || HALF == 32, "half a row of the head dim");
            uint32_t v[HALF];   // both TMEM loads of a half row in flight together
            tmem_ld32(tm + tq + 128 + hh * HALF, *reinterpret_cast<uint32_t(*)[32]>(v));
            if (HALF == 64) tmem_ld32(tm + tq + 128 + hh * HALF + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * (HALF / 64)));
            tmem_ld_wait();
            if (has64) {
                const int rr = D + t;
#pragma unroll
                for (int cc = 0; cc < HALF / 8; ++cc) {
                    const int col = hh * HALF + 8 * cc;
                    *reinterpret_cast<uint4 *>(sEst + (col >> 6) * (R * 128) + rr * 128 +
                                               ((((col & 63) >> 3) ^ (rr & 7)) << 4)) = pack8u(v + 8 * cc);
                }
            }
            tmem_ld32(tm + tq + hh * HALF, *reinterpret_cast<uint32_t(*)[32]>(v));
            if (HALF == 64) tmem_ld32(tm + tq + hh * HALF + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * (HALF / 64)));
            tmem_ld_wait();
            if (has_row) {   // E[i][j] = gamma_C delta_ij - (K~^T W)[i][j]
                // the diagonal lies in this half for the warps whose rows are its rows (warp-uniform)
                const bool dhalf = (i / HALF) == hh;
#pragma unroll
                for (int cc = 0; cc < HALF / 8; ++cc) {
                    const int col = hh * HALF + 8 * cc;
                    uint4 w;
                    if (dhalf) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[e] = (col + e == i ? gamma_c : 0.f) - __uint_as_float(v[8 * cc + e]);
                        w = pack8(f);
                    } else {
                        w = pack8un(v + 8 * cc);
                    }
                    *reinterpret_cast<uint4 *>(sEst + (col >> 6) * (R * 128) + i * 128 +
                                               ((((col & 63) >> 3) ^ (i & 7)) << 4)) = w;
                }
            }
        }

        fence_proxy_async();
        tc_fence_before();
        named_sync(bar, kGroupThreads);
        const bool failed = ctl->fail != 0;
        if (tid == 0 && failed) record_error(p.ws, 1);
        if (tid == kStoreThread && !failed) {   // stored once the next chunk has started
            staged = cur.slot;
            staged_col = cur.col;
        }
        if (!more || failed) break;
        cur = nx;
    }
    cp_async_wait_all();
    if (tid == kStoreThread) {   // the last chunk's state columns; shared memory must outlive the stores
        if (staged >= 0) {
            for (int kb = 0; kb < NB; ++kb)
                tma_store_3d(map_E, sEst + kb * (R * 128), kb * 64, 0, staged);
            bulk_commit();
        }
        bulk_wait0();
        if (pend >= 0) release_slot(p, pend, pend_col);
        if (staged >= 0) release_slot(p, staged, staged_col);
    }
}

// ---------------------------------------------------------------------------------
// prep with a decay per key channel (TileOPs KDAFwdOp: g [.., K]; GLARecurrentFwdOp:
// diag(exp(gk)) applied to the state).  E_c keeps its form; the decays become diagonal
// per channel.  With G_t[c] the in-chunk cumulative log decay of channel c (inclusive),
// R_t = G_t when the delta term reads the decayed state and G_{t-1} otherwise, and
//   K_R = [k^_t * exp(R_t)],  Q_G = [q~_t * exp(G_t)],  K~ = [k^_s * exp(G_n - G_s)]
// ("*" elementwise, rows t), P = T diag(beta):
//
//   L[t][s]   = beta_t sum_c k^_t[c] k^_s[c] exp(R_t[c] - G_s[c])   (s < t),  T = (I + L)^{-1}
//   Aqk[t][s] = sum_c q~_t[c] k^_s[c] exp(G_t[c] - G_s[c])          (s <= t)
//   [ S_next ]   [ diag(exp G_n) - Z1 K_R   Z1 ] [ S ]
//   [   O    ] = [ Q_G - Z2 K_R             Z2 ] [ V ],    Z1 = K~^T P,  Z2 = Aqk P
//
// (W = P K_R is never formed: Z1 K_R = K~^T W and Z2 K_R = Aqk W.)  The factor inside L
// and Aqk is split over 16-token sub-blocks, the sub-chunk form of the kda-neuron-kernels
// README: for rows t of sub-block b and G_ref the cumulative decay at the token before it,
//   exp(R_t - G_s) = exp(R_t - G_ref) exp(G_ref - G_s),
// so the Gram rows of sub-block b are one tensor-core product of two scaled copies of k
// and q.  The row factor is <= 1, and so is the column factor of every earlier sub-block;
// only the sub-block's own columns get a factor above 1, up to exp of its 16-token decay.
// When that span passes kSpanLog2 in some channel, the sub-block's diagonal entries are
// recomputed on CUDA cores with the exact factor per element, so the result is exact for
// any decay.  One group per CTA, of all 512 threads (the scaled copies take the shared
// memory a second group would need); E_c goes to global memory by ordinary stores from
// the epilogues.
// ---------------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSpanLog2 = 60.f * kLog2e;    // sub-block spans above e^60 take the exact path
constexpr float kClampLog2 = 100.f;           // keeps the factors of such a sub-block finite

template <int D>
struct GkSmem {
    static constexpr int NB = D / 64;
    static constexpr int KQ = 0;                          // raw [K;Q]: NB x 16 KB, K-major SW128
    static constexpr int KRQG = KQ + NB * 16384;          // [K_R; Q_G], same layout
    static constexpr int KT = KRQG + NB * 16384;          // K~: NB x 8 KB
    static constexpr int GF = KT + NB * 8192;             // g, then G in log2 units: fp32 [64][D]
    static constexpr int OV = GF + 64 * D * 4;            // Gram operands; later L, T | P | Aqk; Z ops
    static constexpr int GA = OV;                         // column operands: NB x 160 rows x 128 B
    static constexpr int GB = GA + NB * 160 * 128;        // row operands: NB x 128 rows x 128 B
    static constexpr int LT_BYTES = 2 * 64 * kLP * 4;     // L and T fp32
    static constexpr int PT = OV + LT_BYTES;              // P: MN-major 64 x 64
    static constexpr int AQ = PT + 8192;                  // Aqk: K-major 64 x 64
    static constexpr int ZOPS = D * 128 + 16384;          // Z1 and [-Z2 | I], from OV, after MMA2
    static constexpr int ST = OV + ZOPS;                  // per-warp E_c staging (epilogues 2, 3): 16 x 2 KB
    static constexpr int OV_A = GB - OV + NB * 128 * 128, OV_B = AQ + 8192 - OV, OV_C = ZOPS + 16 * 2048;
    static constexpr int OV_BYTES = OV_A > OV_B ? (OV_A > OV_C ? OV_A : OV_C) : (OV_B > OV_C ? OV_B : OV_C);
    static constexpr int SD = OV + OV_BYTES;              // exact diagonal sub-blocks: fp32 [4][2][16][16]
    static constexpr int MISC = SD + 4 * 2 * 256 * 4;
    // MISC: beta [2][64] | kn [64] | qn [64] | exp(G_n) [D] | prefix totals [1024] | span flags [4]
    //       | gate parameters: A_log, pad [3], dt_bias [D]
    static constexpr int CTRL = MISC + (2 * 64 + 64 + 64 + D + 1024 + 4 + 4 + D) * 4;
    static constexpr int BYTES = ((CTRL + 64 + 1023) / 1024) * 1024;
};

// A warp's rows of E_c (lane l holds row row0 + l, l < nrows = 16 or 32; 32 fp32 values
// in u for columns col0 ..) go to global memory by TMA stores of 16-row x 32-column boxes
// from a 2 KB staging tile of the warp, laid out in the 64-byte swizzle of the tensor map
// (16-byte chunk c of row r at position c ^ ((r >> 1) & 3): conflict-free writes).  The
// stores stay in flight: lane 0 waits for them (bulk_wait0) before E_c is published, and
// every call first waits until the tile's previous store has read it.  With neg the values
// are negated and dval added at column dcol (relative to col0; none when outside 0..31).
__device__ __forceinline__ void warp_store_E(uint8_t *stage, const CUtensorMap *map, int slot, int row0,
                                             int nrows, int col0, const uint32_t *u, bool neg, int lane,
                                             bool issue, int dcol = -1, float dval = 0.f) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 w;
        if (neg) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = (8 * c + e == dcol ? dval : 0.f) - __uint_as_float(u[8 * c + e]);
            w = pack8(f);
        } else {
            w = pack8u(u + 8 * c);
        }
        *reinterpret_cast<uint4 *>(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = w;
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0 && issue) {
        fence_proxy_async_global();   // after the slot's acquire (wait_slot_free) in another thread
        tma_store_3d(map, stage, col0, row0, slot);
        if (nrows == 32) tma_store_3d(map, stage + 1024, col0, row0 + 16, slot);
        bulk_commit();
    }
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// g of one chunk (fp32 rows, zero past the chunk's valid tokens) by 16-byte cp.async copies
// (threads 0..255 without warps 0 and 4, as load_rows)
template <int D>
__device__ __forceinline__ void load_g(const TcParams &p, float *gf, const ChunkItem &it, int tid) {
    constexpr int PPR = D / 4;
    const int w = tid >> 5;
    if (w == 0 || w == 4) return;
    const int lt = (w < 4 ? tid - 32 : tid - 64);
    for (int pidx = lt; pidx < 64 * PPR; pidx += kGroupThreads - 64) {
        const int row = pidx / PPR, pc = pidx % PPR;
        const bool in = row < it.nv;
        const float *src = p.gk + ((it.row0 + (in ? row : 0)) * p.H + it.h) * D + 4 * pc;
        cp_async16(gf + row * D + 4 * pc, src, in ? 16u : 0u);
    }
    cp_async_commit();
}
__device__ __forceinline__ void load_beta(const TcParams &p, float *mbeta, const ChunkItem &it, int tid) {
    const int t = tid - 64;   // warps 2, 3
    if (t >= 0 && t < 64) {
        const long gi = (it.row0 + (t < it.nv ? t : 0)) * p.H + it.h;
        cp_async4(mbeta + t, p.beta + gi, t < it.nv ? 4u : 0u);
    }
    cp_async_commit();
}
// A_log and dt_bias [D] of the chunk's head for a raw-gate g (warps 1-3), ahead of the prefix
template <int D>
__device__ __forceinline__ void load_gate(const TcParams &p, float *gate, const ChunkItem &it, int tid) {
    if (!p.A_log || tid < 32 || tid >= 128) return;
    for (int c = tid - 32; c <= D; c += 96) {
        if (c == D) cp_async4(gate, p.A_log + it.h, 4u);
        else cp_async4(gate + 4 + c, p.dt_bias ? p.dt_bias + (size_t)it.h * D + c : p.A_log, p.dt_bias ? 4u : 0u);
    }
    cp_async_commit();
}

constexpr int kGkThreads = 512;   // the whole CTA: one prep group
constexpr int kGkBarInv = 2;      // named barrier of the inverse (threads 0..255)
constexpr int kGkBarPark = 3;     // threads 256..511 wait there while the inverse runs

// OPT: the gate and beta prologues and grouped heads (the decayed read is always a runtime choice)
template <int D, bool OPT>
__device__ __forceinline__ void prep_group_gk(const CUtensorMap *map_Ew, const TcParams &p, uint8_t *sm,
                                              uint32_t tm, int tid, int bar) {
    using Ly = GkSmem<D>;
    constexpr int NT = kGkThreads;
    constexpr int NB = D / 64;
    constexpr int NP = D / 2;                 // channel pairs
    constexpr int NQ = NT / NP;               // token groups of the prefix and the build
    constexpr int TPG = 64 / NQ;              // their tokens: 8 (D = 128) or 4 (D = 64)
    static_assert(TPG <= 16 && 16 % TPG == 0, "a token group stays inside one 16-token sub-block");
    PrepCtrl *ctl = reinterpret_cast<PrepCtrl *>(sm + Ly::CTRL);
    __shared__ uint32_t s_seen_gk[kMaxChains];   // the ring counters last read
    uint32_t *seen = s_seen_gk;
    if (tid < kMaxChains) seen[tid] = 0;         // (first read after the loop's barriers)
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hh = warp >> 2;   // TMEM lane quadrant; column quarter
    const int i128 = 32 * q4 + lane;
    const int i64 = 16 * q4 + lane;
    const bool has64 = lane < 16;
    const uint32_t tq = (uint32_t)(32 * q4) << 16;
    const bool loader = tid < kGroupThreads;   // load_rows, load_g, load_beta use threads 0..255

    uint8_t *sKQ = sm + Ly::KQ;
    uint8_t *sKR = sm + Ly::KRQG;
    uint8_t *sKT = sm + Ly::KT;
    float *gf = reinterpret_cast<float *>(sm + Ly::GF);
    uint8_t *sGA = sm + Ly::GA;
    uint8_t *sGB = sm + Ly::GB;
    float *sL = reinterpret_cast<float *>(sm + Ly::OV);
    float *sT = sL + 64 * kLP;
    uint8_t *sP = sm + Ly::PT;
    uint8_t *sA = sm + Ly::AQ;
    uint8_t *sZ1 = sm + Ly::OV;                 // after MMA2: Z1 (K-major D x 64)
    uint8_t *sZ2 = sm + Ly::OV + D * 128;       // [-Z2 | I] (K-major 64 x 128)
    static_assert(D * 128 + 16384 <= 2 * 64 * kLP * 4, "the Z operands overlay L and T only");
    uint8_t *stage = sm + Ly::ST + warp * 2048;
    float *sd = reinterpret_cast<float *>(sm + Ly::SD);
    float *mbeta2 = reinterpret_cast<float *>(sm + Ly::MISC);
    float *mkn = mbeta2 + 128, *mqn = mkn + 64, *meGn = mqn + 64, *mtot = meGn + D;
    int *mspan = reinterpret_cast<int *>(mtot + 1024);
    float *mgate = reinterpret_cast<float *>(mspan + 4);   // A_log, pad, dt_bias [D] at +4

    const long n_items = prep_items(p);
    if (tid == 0) ctl->more = claim_item(p, n_items, ctl->nxi);
    named_sync(bar, NT);
    if (!ctl->more) return;
    ChunkItem cur = ctl->nxi;
    named_sync(bar, NT);   // everyone has read the item before it is claimed again
    if (tid == 0) ctl->more = claim_item(p, n_items, ctl->nxi);   // the next chunk, read after the barrier below
    named_sync(bar, NT);
    if (loader) {
        load_rows<D, OPT>(p, sKQ, cur, tid, true);
        load_rows<D, OPT>(p, sKQ, cur, tid, false);
        load_g<D>(p, gf, cur, tid);
        load_beta(p, mbeta2, cur, tid);
        if (OPT) load_gate<D>(p, mgate, cur, tid);
    }
    int pend = -1, pend_col = 0;   // kStoreThread: slot (column) whose E_c stores are issued, not published
    const bool decayed = p.decayed_read != 0;

    for (uint32_t it = 0;; ++it) {
        const uint32_t ph = it & 1;
        const int nv = cur.nv;
        float *mbeta = mbeta2 + 64 * (it & 1);
        if (tid < 4) mspan[tid] = 0;
        const bool gate = OPT && p.A_log != nullptr;   // g holds the raw gate
        cp_async_wait_all();
        if (lane == 0) bulk_wait0();   // the previous chunk's E_c stores: complete, staging free
        named_sync(bar, NT);
        bool ok = ctl->fail == 0;

        // ---- norms of the k and q rows (zero past the valid tokens), four threads a row;
        // prefix over tokens of g
        {
            const int r = tid >> 2, part = tid & 3, t = r & 63;
            const bool isq = r >= 64;
            float ss = 0.f;
#pragma unroll
            for (int cc = 0; cc < NB * 2; ++cc) {
                const int chunk = part * NB * 2 + cc;
                const uint4 w = *reinterpret_cast<const uint4 *>(sKQ + (chunk >> 3) * 16384 + (isq ? 8192 : 0) +
                                                                 t * 128 + (((chunk ^ t) & 7) << 4));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = bf16lo(ws[e]), b = bf16hi(ws[e]);
                    ss = fmaf(a, a, fmaf(b, b, ss));
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            if (part == 0) {
                const float inv = p.use_l2 ? 1.f / fmaxf(sqrtf(ss), kNormEps) : 1.f;
                if (isq) mqn[t] = t < nv ? p.scale * inv : 0.f;
                else mkn[t] = t < nv ? inv : 0.f;
            }
            if (OPT && p.beta_sig && tid >= 448)   // beta from logits (zero past the valid tokens)
                mbeta[tid - 448] = tid - 448 < nv ? beta_of(mbeta[tid - 448], 1, p.neg_eig) : 0.f;
        }
        {   // pass A: each token group's inclusive prefix in place (a channel pair per thread),
            // in log2 units
            const int c0 = 2 * (tid % NP), j = tid / NP;
            float2 acc = make_float2(0.f, 0.f);
            const float gate_a = gate ? expf(mgate[0]) : 0.f;
            const float2 gate_bi = gate ? *reinterpret_cast<const float2 *>(mgate + 4 + c0) : make_float2(0.f, 0.f);
#pragma unroll
            for (int t = j * TPG; t < (j + 1) * TPG; ++t) {
                float2 *x = reinterpret_cast<float2 *>(gf + t * D + c0);
                float2 gv = *x;
                if (gate) {   // g holds the raw gate
                    gv.x = t < nv ? gate_decay_a(gv.x, gate_a, gate_bi.x) : 0.f;
                    gv.y = t < nv ? gate_decay_a(gv.y, gate_a, gate_bi.y) : 0.f;
                }
                acc.x = fmaf(gv.x, kLog2e, acc.x);
                acc.y = fmaf(gv.y, kLog2e, acc.y);
                *x = acc;
            }
            *reinterpret_cast<float2 *>(mtot + j * D + c0) = acc;
        }
        named_sync(bar, NT);
        {   // pass B: add the totals of the earlier groups
            const int c0 = 2 * (tid % NP), j = tid / NP;
            float2 off = make_float2(0.f, 0.f);
            for (int jj = 0; jj < j; ++jj) {
                const float2 tv = *reinterpret_cast<const float2 *>(mtot + jj * D + c0);
                off.x += tv.x;
                off.y += tv.y;
            }
            if (j > 0) {
#pragma unroll
                for (int t = j * TPG; t < (j + 1) * TPG; ++t) {
                    float2 *x = reinterpret_cast<float2 *>(gf + t * D + c0);
                    const float2 gv = *x;
                    *x = make_float2(gv.x + off.x, gv.y + off.y);
                }
            }
        }
        named_sync(bar, NT);

        // ---- build: K~, [K_R; Q_G] and the sub-block Gram operands, channel pair cp of
        // tokens [t0, t0 + TPG) (all inside sub-block b).  Per token three exponentials of
        // each channel, fq = e^(G_t - G_ref(b)) <= 1, fb = e^(G_ref(b) - G_t) >= 1 and
        // f1 = e^(G_ref(b+1) - G_t) <= 1 (G_ref(4) := G_n); every other factor is one of
        // these times a per-thread constant <= 1.
        {
            const int cp = tid % NP, c0 = 2 * cp;
            const int t0 = (tid / NP) * TPG, b = t0 >> 4;
            float2 gref[5];
#pragma unroll
            for (int bb = 0; bb < 5; ++bb)
                gref[bb] = bb == 0 ? make_float2(0.f, 0.f)
                                   : *reinterpret_cast<const float2 *>(gf + (bb == 4 ? 63 : 16 * bb - 1) * D + c0);
            float2 grb = gref[0], grb1 = gref[1];
#pragma unroll
            for (int bb = 1; bb < 4; ++bb)
                if (bb == b) { grb = gref[bb]; grb1 = gref[bb + 1]; }
            const float2 gn = gref[4];
            if (t0 == 0) {
                meGn[c0] = ex2f(gn.x);
                meGn[c0 + 1] = ex2f(gn.y);
            }
            if ((t0 & 15) == 0) {   // span of sub-block b in these two channels
                const float2 ge = *reinterpret_cast<const float2 *>(gf + (16 * b + 15) * D + c0);
                if (fmaxf(grb.x - ge.x, grb.y - ge.y) > kSpanLog2) atomicOr(mspan + b, 1);
            }
            const float eb0 = ex2f(grb.x), eb1 = ex2f(grb.y);               // e^G_ref(b)
            const float cn0 = ex2f(gn.x - grb1.x), cn1 = ex2f(gn.y - grb1.y);  // e^(G_n - G_ref(b+1))
            float cb0[4], cb1[4];                                              // e^(G_ref(b') - G_ref(b+1))
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                cb0[bb] = ex2f(gref[bb].x - grb1.x);
                cb1[bb] = ex2f(gref[bb].y - grb1.y);
            }
            float fqp0 = 1.f, fqp1 = 1.f;   // fq of the previous token (1 before the sub-block)
            if ((t0 & 15) != 0) {
                const float2 gp = *reinterpret_cast<const float2 *>(gf + (t0 - 1) * D + c0);
                fqp0 = ex2f(gp.x - grb.x);
                fqp1 = ex2f(gp.y - grb.y);
            }
#pragma unroll
            for (int t = t0; t < t0 + TPG; ++t) {
                const float2 g = *reinterpret_cast<const float2 *>(gf + t * D + c0);
                const uint32_t kw = *reinterpret_cast<const uint32_t *>(sKQ + kmajor_sw128_offset(128, t, c0));
                const uint32_t qw = *reinterpret_cast<const uint32_t *>(sKQ + kmajor_sw128_offset(128, 64 + t, c0));
                const float kn = mkn[t], qn = mqn[t];
                const float k0 = bf16lo(kw) * kn, k1 = bf16hi(kw) * kn;
                const float qa = bf16lo(qw) * qn, qb = bf16hi(qw) * qn;
                const float fq0 = ex2f(g.x - grb.x), fq1 = ex2f(g.y - grb.y);
                const float fb0 = ex2f(fminf(grb.x - g.x, kClampLog2)), fb1 = ex2f(fminf(grb.y - g.y, kClampLog2));
                const float f10 = ex2f(grb1.x - g.x), f11 = ex2f(grb1.y - g.y);
                const float fk0 = decayed ? fq0 : fqp0, fk1 = decayed ? fq1 : fqp1;
                *reinterpret_cast<uint32_t *>(sKT + kmajor_sw128_offset(64, t, c0)) =
                    pack_bf16(k0 * f10 * cn0, k1 * f11 * cn1);
                *reinterpret_cast<uint32_t *>(sKR + kmajor_sw128_offset(128, t, c0)) =
                    pack_bf16(k0 * fk0 * eb0, k1 * fk1 * eb1);
                *reinterpret_cast<uint32_t *>(sKR + kmajor_sw128_offset(128, 64 + t, c0)) =
                    pack_bf16(qa * fq0 * eb0, qb * fq1 * eb1);
                // row operands of sub-block b: k rows 32b + j, q rows 32b + 16 + j
                const int j = t - 16 * b;
                *reinterpret_cast<uint32_t *>(sGB + kmajor_sw128_offset(128, 32 * b + j, c0)) =
                    pack_bf16(k0 * fk0, k1 * fk1);
                *reinterpret_cast<uint32_t *>(sGB + kmajor_sw128_offset(128, 32 * b + 16 + j, c0)) =
                    pack_bf16(qa * fq0, qb * fq1);
                // column operands of sub-blocks b' >= b: row off(b') + t, factor e^(G_ref(b') - G_t)
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    if (bb < b) continue;
                    const int off = bb == 0 ? 0 : (bb == 1 ? 16 : (bb == 2 ? 48 : 96));
                    const float f0 = bb == b ? fb0 : f10 * cb0[bb];
                    const float f1 = bb == b ? fb1 : f11 * cb1[bb];
                    *reinterpret_cast<uint32_t *>(sGA + kmajor_sw128_offset(160, off + t, c0)) =
                        pack_bf16(k0 * f0, k1 * f1);
                }
                fqp0 = fq0;
                fqp1 = fq1;
            }
        }
        fence_proxy_async();
        named_sync(bar, NT);

        // ---- sub-blocks whose decay span is too wide for the split: exact diagonal entries
        for (int b = 0; b < 4; ++b) {
            if (mspan[b] == 0 || tid >= 256) continue;   // mspan: uniform, read after the barrier
            const int tj = tid >> 4, sj = tid & 15, t = 16 * b + tj, s = 16 * b + sj;
            float aq = 0.f, al = 0.f;
            if (sj <= tj) {
                for (int c = 0; c < D; ++c) {
                    const float kt = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                         sKQ + kmajor_sw128_offset(128, t, c))) * mkn[t];
                    const float qt = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                         sKQ + kmajor_sw128_offset(128, 64 + t, c))) * mqn[t];
                    const float ks = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                                         sKQ + kmajor_sw128_offset(128, s, c))) * mkn[s];
                    const float gt = gf[t * D + c], gs = gf[s * D + c];
                    const float rt = decayed ? gt : (t == 0 ? 0.f : gf[(t - 1) * D + c]);
                    aq = fmaf(qt * ks, ex2f(gt - gs), aq);
                    if (sj < tj) al = fmaf(kt * ks, ex2f(rt - gs), al);
                }
            }
            sd[(b * 2 + 0) * 256 + tj * 16 + sj] = al;
            sd[(b * 2 + 1) * 256 + tj * 16 + sj] = aq;
        }
        if (mspan[0] | mspan[1] | mspan[2] | mspan[3]) named_sync(bar, NT);

        // ---- MMA1: sub-block b's Gram rows, transposed: D1[s][32 b + j] for s < 16 (b + 1):
        // column operand rows s (M = 64), row operand k rows then q rows of sub-block b (N = 32)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t id = idesc_bf16_f32(64, 32, false, false);
            const uint32_t ga = smem_u32(sGA), gb = smem_u32(sGB);
            for (int b = 0; b < 4; ++b) {
                const int off = b == 0 ? 0 : (b == 1 ? 16 : (b == 2 ? 48 : 96));
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_bf16_ss(tm + 32 * b, desc_kmajor_sw128(ga + off * 128, 160, ks),
                                desc_kmajor_sw128(gb + 32 * b * 128, 128, ks), id, ks > 0 ? 1u : 0u);
            }
            mma_commit(&ctl->bar_mma);
        }
        // raw q, k and g are no longer read: the next chunk's loads start once MMA1 is issued
        // (packed sequences read cu_seqlens to find it: off the path to MMA1)
        // the next chunk: claimed by thread 0 before the previous barrier, read here by all,
        // claimed again after epilogue 1's barrier
        const bool more = ctl->more != 0;
        const ChunkItem nx = ctl->nxi;
        float *mbeta_next = mbeta2 + 64 * ((it + 1) & 1);
        if (ok && more && loader) {
            load_rows<D, OPT>(p, sKQ, nx, tid, true);
            load_rows<D, OPT>(p, sKQ, nx, tid, false);
            load_g<D>(p, gf, nx, tid);
            load_beta(p, mbeta_next, nx, tid);
            if (OPT) load_gate<D>(p, mgate, nx, tid);
        }

        if (tid == kStoreThread && pend >= 0) {   // the previous chunk's E_c, while MMA1 runs
            release_slot(p, pend, pend_col);
            pend = -1;
        }
        // this chunk's ring slot must have been read by its chain before epilogue 2 stores
        // into it (the barriers in between order every warp's stores after this wait)
        if (tid == kStoreThread && ok && !wait_slot_free(p, cur.chain, cur.col, kWaitNs, seen)) {
            ctl->fail = 1;
            record_error(p.ws, 4);
        }
        if (ok && !mbar_wait(&ctl->bar_mma, ph, kWaitNs)) ctl->fail = 1;
        tc_fence_after();

        // ---- epilogue 1: L (fp32, rows t) and Aqk (bf16 operand) from the transposed rows s;
        // the warps of column quarter hh take sub-block b = hh
        {
            const int s = i64, bs = s >> 4, b = hh;
            uint32_t v[32];
            tmem_ld32(tm + tq + 32 * b, v);
            tmem_ld_wait();
            if (has64) {
                const bool exact = mspan[b] != 0 && bs == b;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = 16 * b + j;
                    float lval = 0.f, aval = 0.f;
                    if (b >= bs) {
                        lval = exact ? sd[(b * 2) * 256 + j * 16 + (s & 15)] : __uint_as_float(v[j]);
                        aval = exact ? sd[(b * 2 + 1) * 256 + j * 16 + (s & 15)] : __uint_as_float(v[16 + j]);
                        lval = s < t ? mbeta[t] * lval : 0.f;
                        aval = s <= t ? aval : 0.f;
                        sL[t * kLP + s] = lval;
                    }
                    *reinterpret_cast<__nv_bfloat16 *>(sA + kmajor_sw128_offset(64, t, s)) =
                        __float2bfloat16_rn(aval);
                }
            }
        }
        fence_proxy_async();
        named_sync(bar, NT);
        ok = ctl->fail == 0;
        // the chunk after next (a thread that waits out the inverse anyway)
        if (tid == kGroupThreads) ctl->more = claim_item(p, n_items, ctl->nxi);

        // ---- T = (I + L)^{-1}, written as P = T diag(beta) (MN-major: row t, columns s), by
        // threads 0..255
        if (tid < kGroupThreads) {
            invert_unit_lower_64<kGroupThreads, true>(sL, sT, BTiles{sP, nullptr, nullptr, mbeta, nullptr},
                                                      tid, kGkBarInv, [] {});
            named_arrive(kGkBarPark, NT);
        } else {
            named_sync(kGkBarPark, NT);   // wait without taking issue slots from the inverse
        }

        // ---- MMA2: D2a[:, 0:64] = K~^T P (M = D);  D2b[:, 128:192] = Aqk P (M = 64)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t ida = idesc_bf16_f32(D, 64, true, true);
            const uint32_t idb = idesc_bf16_f32(64, 64, false, true);
            const uint32_t kt = smem_u32(sKT), pp = smem_u32(sP), aa = smem_u32(sA);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm, desc_mnmajor_sw128(kt, 64, ks), desc_mnmajor_sw128(pp, 64, ks), ida,
                            ks > 0 ? 1u : 0u);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm + 128, desc_kmajor_sw128(aa, 64, ks), desc_mnmajor_sw128(pp, 64, ks), idb,
                            ks > 0 ? 1u : 0u);
            mma_commit(&ctl->bar_mma);
        }
        if (ok && !mbar_wait(&ctl->bar_mma, ph ^ 1u, kWaitNs)) ctl->fail = 1;
        tc_fence_after();

        // ---- epilogue 2: column quarters 0, 1 take Z1 = D2a (-> E[i][D + s], MMA3a's A),
        // quarters 2, 3 take Z2 = D2b (-> E[D + t][D + s], MMA3b's A = [-Z2 | I])
        const int slot = cur.slot;
        constexpr int RW = D == 128 ? 32 : 16;   // rows of an M = D result per warp
        if (hh < 2) {
            uint32_t v[32];
            tmem_ld32(tm + tq + 32 * hh, v);
            tmem_ld_wait();
            const bool has_row = (D == 128) || has64;
            const int i = (D == 128) ? i128 : i64;
            if (has_row) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = 32 * hh + 8 * cc;
                    *reinterpret_cast<uint4 *>(sZ1 + i * 128 + ((((col >> 3) ^ i) & 7) << 4)) = pack8u(v + 8 * cc);
                }
            }
            warp_store_E(stage, map_Ew, slot, RW * q4, RW, D + 32 * hh, v, false, lane, ok);
        } else {
            const int hq = hh - 2;
            uint32_t v[32];
            tmem_ld32(tm + tq + 128 + 32 * hq, v);
            tmem_ld_wait();
            const int t = i64;
            if (has64) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int col = 32 * hq + 8 * cc;
                    const int off = t * 128 + ((((col >> 3) ^ t) & 7) << 4);
                    *reinterpret_cast<uint4 *>(sZ2 + off) = pack8un(v + 8 * cc);
                    float dg[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) dg[e] = (col + e == t) ? 1.f : 0.f;
                    *reinterpret_cast<uint4 *>(sZ2 + 8192 + off) = pack8(dg);
                }
            }
            warp_store_E(stage, map_Ew, slot, D + 16 * q4, 16, D + 32 * hq, v, false, lane, ok);
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(bar, NT);
        ok = ctl->fail == 0;

        // ---- MMA3: D3a[:, 0:D] = Z1 K_R (M = D);  D3b[:, 128:128+D] = [-Z2 | I] [K_R; Q_G] (M = 64)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t ida = idesc_bf16_f32(D, D, false, true);
            const uint32_t idb = idesc_bf16_f32(64, D, false, true);
            const uint32_t kr = smem_u32(sKR), z1 = smem_u32(sZ1), z2 = smem_u32(sZ2);
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(tm, desc_kmajor_sw128(z1, D, ks), desc_mnmajor_sw128(kr, 128, ks), ida,
                            ks > 0 ? 1u : 0u);
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ss(tm + 128, desc_kmajor_sw128(z2, 64, ks), desc_mnmajor_sw128(kr, 128, ks), idb,
                            ks > 0 ? 1u : 0u);
            mma_commit(&ctl->bar_mma);
        }
        if (ok && !mbar_wait(&ctl->bar_mma, ph, kWaitNs)) ctl->fail = 1;
        tc_fence_after();

        // ---- epilogue 3: the state columns of E, 32 columns per warp.
        //   E[D + t][j] = Q_G[t][j] - (Z2 K_R)[t][j] = D3b[t][j]
        //   E[i][j]     = exp(G_n[i]) delta_ij - (Z1 K_R)[i][j]
        {
            uint32_t v[32];
            if constexpr (D == 128) {
                tmem_ld32(tm + tq + 128 + 32 * hh, v);
                tmem_ld_wait();
                warp_store_E(stage, map_Ew, slot, D + 16 * q4, 16, 32 * hh, v, false, lane, ok);
                tmem_ld32(tm + tq + 32 * hh, v);
                tmem_ld_wait();
                warp_store_E(stage, map_Ew, slot, 32 * q4, 32, 32 * hh, v, true, lane, ok, i128 - 32 * hh,
                             meGn[i128]);
            } else if (hh < 2) {
                tmem_ld32(tm + tq + 32 * hh, v);
                tmem_ld_wait();
                warp_store_E(stage, map_Ew, slot, 16 * q4, 16, 32 * hh, v, true, lane, ok, i64 - 32 * hh,
                             has64 ? meGn[i64] : 0.f);
            } else {
                tmem_ld32(tm + tq + 128 + 32 * (hh - 2), v);
                tmem_ld_wait();
                warp_store_E(stage, map_Ew, slot, D + 16 * q4, 16, 32 * (hh - 2), v, false, lane, ok);
            }
        }
        tc_fence_before();
        named_sync(bar, NT);   // every warp's E_c stores are issued
        const bool failed = ctl->fail != 0;
        if (tid == 0 && failed) record_error(p.ws, 2);
        if (tid == kStoreThread && !failed) {
            pend = cur.slot;
            pend_col = cur.col;
        }
        if (!more || failed) break;
        cur = nx;
    }
    cp_async_wait_all();
    if (lane == 0) bulk_wait0();   // the last chunk's E_c stores have completed ...
    named_sync(bar, NT);           // ... in every warp, before it is published
    if (tid == kStoreThread && pend >= 0) release_slot(p, pend, pend_col);
}

// ---------------------------------------------------------------------------------
// chain -- one CTA per (sequence, head), transposed so that M = dv:
//
//   D^T[j][r] = sum_k A[j][k] E_c[r][k],   A = [S^T | V_c^T]   (dv rows, D + 64 columns)
//
// hence D^T[j][r] = S_next[r][j] for r < D and O[r - D][j] for r >= D: the next
// state and the chunk's outputs come out of the same instructions.  The V half
// (4 k-steps) needs only E_c and V_c, so it is issued into the next of two TMEM
// accumulators while the epilogue of the previous chunk is still running; only the
// state half (D / 16 k-steps) waits for S_c.  A tcgen05 MMA of M = 128 costs about
// the same per k-step for any N up to 128-192, which is why the whole head (and
// its outputs) is one wide product rather than several narrow ones.
// The state is carried as the bf16 operand S^T, rebuilt every chunk from the fp32
// accumulator; the final state is stored from the fp32 accumulator.
// Warps: 0 producers, 1 MMA, 2..9 state epilogue (two per TMEM lane quadrant, one
// half of the state columns each), 10..13 output epilogue; any others idle.
// ---------------------------------------------------------------------------------
template <int D>
struct ChainCfg {
    static constexpr int R = D + 64;              // rows / columns of E_c
    static constexpr int NKB = R / 64;            // 64-wide K blocks of E_c
    static constexpr int NB = D / 64;             // 64-wide blocks of the head dim
    static constexpr int E_BYTES = R * R * 2;     // one stage of E_c (K-major SW128, R rows)
    static constexpr int AS_BYTES = D * D * 2;    // S^T operand (K-major SW128, D rows)
    static constexpr int AV_BYTES = 64 * D * 2;   // one stage of V_c (MN-major SW128)
    static constexpr int O_BYTES = 64 * D * 2;    // output staging [64][D] bf16
    static constexpr int SMEM = 2 * E_BYTES + AS_BYTES + 2 * AV_BYTES + O_BYTES + 1024;
    static constexpr uint32_t TCOLS = (2 * R <= 256) ? 256u : 512u;   // two accumulators
};

// One task of a chain CTA: the (sequence, head) of round r, or none past the last task.
struct ChainTask {
    long start;   // first token row
    int len, nc;  // tokens, chunks
    int n, h;     // sequence, head
    int col0;     // column of its first chunk (round_start of its round)
    int col_end;  // round_start of the next round
};
__device__ __forceinline__ bool chain_task(const TcParams &p, int chain, int r, ChainTask &t) {
    if (r >= p.rounds) return false;
    const int task = r * p.nch + chain;
    if (task >= p.ntask) return false;
    task_info(p, task, t.n, t.h);
    seq_info(p, t.n, t.start, t.len);
    t.nc = (t.len + kC - 1) / kC;
    t.col0 = round_start(p, r);
    t.col_end = round_start(p, r + 1);
    return true;
}

// REV: the reverse walk of the backward, [dS_c; dV_c] = E_c^T [dS_{c+1}; dO_c] (E_c^T's
// product is the same instruction sequence with E_c read MN-major): chunks last to first,
// map_v streams dO, h0 holds the final-state gradient and hT receives the initial-state
// gradient, the "outputs" are the fp32 value gradients (dv_out, or none), and `states` receives
// the incoming state gradient of every chunk.  The maps were kept by a forward launch
// (every chunk its own slot), so nothing waits on flags.
template <int D, bool OPT, bool REV = false>
__device__ __forceinline__ void chain_body(const CUtensorMap *map_E, const CUtensorMap *map_v,
                                           const TcParams &p, uint8_t *sm, int chain) {
    using Cf = ChainCfg<D>;
    constexpr int R = Cf::R;
    constexpr int HALF = D / 2;
    uint8_t *sE0 = sm;
    uint8_t *sAS = sm + 2 * Cf::E_BYTES;
    uint8_t *sAV0 = sAS + Cf::AS_BYTES;
    uint8_t *sO = sAV0 + 2 * Cf::AV_BYTES;
    // s_lo, s_hi: the two K halves of the S^T operand (state rows [0, D/2) and [D/2, D))
    __shared__ uint64_t e_full[2], e_empty[2], v_full[2], v_empty[2], d_full[2], d_free[2], s_lo, s_hi;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_fail;
    // the chain's progress through the ring, as the MMA issuer observes the E_c loads land:
    // every column below s_rel has been loaded (monotone; published by warp 14)
    __shared__ volatile uint32_t s_rel;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&e_full[s], 1);
            mbar_init(&e_empty[s], 1);     // released by the MMA commit
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);     // released by the MMA commit
            mbar_init(&d_full[s], 1);
            mbar_init(&d_free[s], 384);    // the state and the output warps read the accumulator
        }
        mbar_init(&s_lo, 256);
        mbar_init(&s_hi, 256);
        fence_mbar_init();
        s_fail = 0;
        s_rel = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, Cf::TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_slot;

    // Every role walks the same tasks and chunks; gc counts the chunks of this CTA's walk
    // (stages, accumulators and mbarrier phases follow it across tasks).
    ChainTask t;
    if (warp == 0) {
        // ---------------- producers: lane 0 streams E_c (after its ring slot's flag is
        // released), lane 1 streams V_c (with L2 prefetches kPrefetch chunks ahead), each
        // into two shared-memory stages freed by the MMA commit
        constexpr int kPrefetch = 4;
        if (lane == 0) {
            int gc = 0;
            for (int r = 0; chain_task(p, chain, r, t) && !s_fail; ++r) {
                for (int c = 0; c < t.nc && !s_fail; ++c, ++gc) {
                    const int s = gc & 1;
                    const int col = t.col0 + (REV ? t.nc - 1 - c : c);
                    const int slot = chain * p.ring + col % p.ring;
                    // E_c published: watched before the stage frees, so that the round trip to
                    // the flag's line (possibly in the other die's L2) overlaps that wait
                    if (!REV && !wait_flag_acquire(p.flags + slot, (uint32_t)col + 1u, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 16);
                        break;
                    }
                    if (gc >= 2 && !mbar_wait(&e_empty[s], ((gc >> 1) - 1) & 1, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 10);
                        break;
                    }
                    mbar_expect_tx(&e_full[s], Cf::E_BYTES);
                    uint8_t *dE = sE0 + s * Cf::E_BYTES;
                    for (int kb = 0; kb < Cf::NKB; ++kb)
                        tma_load_3d(dE + kb * (R * 128), map_E, &e_full[s], kb * 64, 0, slot);
                }
            }
        } else if (lane == 1) {
            int gc = 0;
            auto chunk_row = [&](int c) { return (int)(t.start + (long)(REV ? t.nc - 1 - c : c) * kC); };
            for (int r = 0; chain_task(p, chain, r, t) && !s_fail; ++r) {
                for (int c = 0; c < kPrefetch && c < t.nc; ++c)
                    for (int mb = 0; mb < Cf::NB; ++mb)
                        tma_prefetch_l2_3d(map_v, mb * 64, t.h, chunk_row(c));
                for (int c = 0; c < t.nc && !s_fail; ++c, ++gc) {
                    const int s = gc & 1;
                    if (gc >= 2 && !mbar_wait(&v_empty[s], ((gc >> 1) - 1) & 1, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 15);
                        break;
                    }
                    mbar_expect_tx(&v_full[s], Cf::AV_BYTES);
                    uint8_t *dV = sAV0 + s * Cf::AV_BYTES;
                    for (int mb = 0; mb < Cf::NB; ++mb)
                        tma_load_3d(dV + mb * 8192, map_v, &v_full[s], mb * 64, t.h, chunk_row(c));
                    if (c + kPrefetch < t.nc)
                        for (int mb = 0; mb < Cf::NB; ++mb)
                            tma_prefetch_l2_3d(map_v, mb * 64, t.h, chunk_row(c + kPrefetch));
                }
            }
        }
    } else if (warp == 14) {
        // ---------------- ring release: publish the chain's progress (s_rel, set by the MMA
        // issuer when an E_c load has landed) to the prep groups by a gpu-scope release,
        // ~900 cycles, kept off the producer and MMA threads.  Only the latest value counts,
        // so a release that falls behind skips ahead.  (The reverse walk has no prep.)
        if (lane == 0 && !REV) {
            uint32_t fin = 0;   // the counter's final value: the end of the chain's last round
            for (int r = 0; chain_task(p, chain, r, t); ++r) fin = (uint32_t)t.col_end;
            uint32_t done = 0;
            uint64_t t0 = globaltimer_ns();
            while (done < fin && !s_fail) {
                const uint32_t v = s_rel;
                if (v > done) {
                    st_release_gpu(p.consumed + chain * kCounterStride, v);
                    done = v;
                    t0 = globaltimer_ns();
                } else if (globaltimer_ns() - t0 > kWaitNs) {
                    s_fail = 1;
                    record_error(p.ws, 17);
                } else {
                    __nanosleep(32);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idV = idesc_bf16_f32(D, R, true, REV);
            const uint32_t idS = idesc_bf16_f32(D, R, false, REV);
            const uint32_t as0 = smem_u32(sAS);
            int gc = 0;
            for (int r = 0; chain_task(p, chain, r, t) && !s_fail; ++r) {
                if (t.nc == 0) s_rel = (uint32_t)t.col_end;   // no chunk: straight to the next round
                for (int c = 0; c < t.nc && !s_fail; ++c, ++gc) {
                    const int b = gc & 1;
                    if (!mbar_wait(&e_full[b], (gc >> 1) & 1, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 11);
                        break;
                    }
                    // E_c of this column is in shared memory: its ring slot may be rewritten
                    // (at the task's last chunk the counter jumps to the next round's start)
                    s_rel = (c + 1 < t.nc) ? (uint32_t)(t.col0 + c + 1) : (uint32_t)t.col_end;
                    if (!mbar_wait(&v_full[b], (gc >> 1) & 1, kWaitNs) ||
                        (gc >= 2 && !mbar_wait(&d_free[b], ((gc >> 1) - 1) & 1, kWaitNs))) {
                        s_fail = 1;
                        record_error(p.ws, 11);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t e0 = smem_u32(sE0 + b * Cf::E_BYTES);
                    const uint32_t av0 = smem_u32(sAV0 + b * Cf::AV_BYTES);
                    const uint32_t dcol = tm + (uint32_t)(b * R);
                    for (int ks = 0; ks < 4; ++ks)   // V half: E_c columns D .. D + 63 (reverse: rows)
                        mma_bf16_ss(dcol, desc_mnmajor_sw128(av0, 64, ks),
                                    REV ? desc_mnmajor_sw128(e0, R, D / 16 + ks) : desc_kmajor_sw128(e0, R, D / 16 + ks),
                                    idV, ks > 0 ? 1u : 0u);
                    // the state half in two K halves: the first D/32 k-steps read state rows
                    // [0, D/2) and start as soon as the epilogue has published them
                    if (!mbar_wait(&s_lo, gc & 1, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 12);
                        break;
                    }
                    tc_fence_after();
                    for (int ks = 0; ks < D / 32; ++ks)   // state half: E_c columns 0 .. D - 1 (reverse: rows)
                        mma_bf16_ss(dcol, desc_kmajor_sw128(as0, D, ks),
                                    REV ? desc_mnmajor_sw128(e0, R, ks) : desc_kmajor_sw128(e0, R, ks), idS, 1u);
                    if (!mbar_wait(&s_hi, gc & 1, kWaitNs)) {
                        s_fail = 1;
                        record_error(p.ws, 12);
                        break;
                    }
                    tc_fence_after();
                    for (int ks = D / 32; ks < D / 16; ++ks)
                        mma_bf16_ss(dcol, desc_kmajor_sw128(as0, D, ks),
                                    REV ? desc_mnmajor_sw128(e0, R, ks) : desc_kmajor_sw128(e0, R, ks), idS, 1u);
                    mma_commit(&d_full[b]);
                    mma_commit(&e_empty[b]);
                    mma_commit(&v_empty[b]);
                }
            }
        }
    } else if (warp < 10) {
        // ---------------- state epilogue, warps 2..9: TMEM quadrant q, value column j.
        // Turns the fp32 next state into the bf16 S^T operand (the critical path) in two
        // halves of the contraction: every warp writes its quarter of state rows [0, D/2)
        // (rows ch D/4 ..), publishes them (s_lo), then its quarter of [D/2, D) (s_hi), so
        // that the next product's first k-steps overlap the second half.  s_lo and s_hi
        // complete once per chunk: after a task's initial state is in place (rows
        // [ch D/2, (ch + 1) D/2) there) and after every chunk but the task's last.
        const int q = warp & 3, ch = (warp - 2) >> 2;
        const bool has_row = (D == 128) || (lane < 16);   // M = 64: 16 rows per quadrant
        const int j = (D == 128) ? 32 * q + lane : 16 * q + lane;
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        const int i_lo = ch * HALF;
        // element (i, j) of a state: key-major at i D + j, value-major at j D + i
        const bool vf = OPT && p.v_first;
        const size_t si = vf ? 1 : D, sj = vf ? D : 1;
        int gc = 0;
        // fp32 state at a chunk's start (key-major [nseq, H, nc, D, D]), kept for the backward
        auto dump_at = [&](int chunk) {
            return p.states + (((size_t)t.n * p.H + t.h) * p.nc_equal + chunk) * D * D;
        };
        for (int r = 0; chain_task(p, chain, r, t) && !s_fail; ++r) {
            const size_t hbase = ((size_t)t.n * p.H + t.h) * D * D;
            if (has_row) {   // S_0^T row j from initial_state[:, j] (the previous task's MMAs are done)
                __nv_bfloat16 *dst = (p.states && t.nc > 0) ? dump_at(REV ? t.nc - 1 : 0) : nullptr;
                for (int i0 = i_lo; i0 < i_lo + HALF; i0 += 8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        x[e] = p.h0 ? p.h0[hbase + (size_t)(i0 + e) * si + j * sj] : 0.f;
                    if (dst)
#pragma unroll
                        for (int e = 0; e < 8; ++e) dst[(size_t)(i0 + e) * D + j] = __float2bfloat16_rn(x[e]);
                    if (t.nc == 0) {
                        if (p.hT)
#pragma unroll
                            for (int e = 0; e < 8; ++e) p.hT[hbase + (size_t)(i0 + e) * si + j * sj] = x[e];
                    } else {
                        const int ci = (i0 & 63) >> 3;
                        *reinterpret_cast<uint4 *>(sAS + (i0 >> 6) * D * 128 + j * 128 + ((ci ^ (j & 7)) << 4)) =
                            make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                       pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
                    }
                }
            }
            if (t.nc == 0) continue;
            fence_proxy_async();
            mbar_arrive(&s_lo);
            mbar_arrive(&s_hi);

            for (int c = 0; c < t.nc; ++c, ++gc) {
                const int b = gc & 1;
                if (s_fail || !mbar_wait(&d_full[b], (gc >> 1) & 1, kWaitNs)) {
                    s_fail = 1;
                    record_error(p.ws, 13);
                    break;
                }
                tc_fence_after();
                constexpr int QP = HALF / 2;   // state rows per warp in each half
                const int i_a = ch * QP, i_b = HALF + ch * QP;   // its rows in [0, D/2), [D/2, D)
                const uint32_t dcol = tm + lrow + (uint32_t)(b * R);
                const bool last = (c + 1 == t.nc);
                uint32_t v[HALF];   // v[0, QP): rows i_a ..; v[QP, 2 QP): rows i_b ..
                if constexpr (QP == 32) {
                    tmem_ld32(dcol + i_a, *reinterpret_cast<uint32_t(*)[32]>(v));
                    tmem_ld32(dcol + i_b, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                } else {
                    tmem_ld16(dcol + i_a, *reinterpret_cast<uint32_t(*)[16]>(v));
                    tmem_ld16(dcol + i_b, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
                }
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&d_free[b]);
                auto store_part = [&](int i0, const uint32_t *vp) {   // QP rows of S^T row j from i0
#pragma unroll
                    for (int cc = 0; cc < QP / 8; ++cc) {
                        const int gcol = (i0 >> 3) + cc;   // 8-column group of S^T row j
                        *reinterpret_cast<uint4 *>(sAS + (gcol >> 3) * D * 128 + j * 128 +
                                                   (((gcol & 7) ^ (j & 7)) << 4)) = pack8u(vp + 8 * cc);
                    }
                };
                if (!last) {
                    if (has_row) store_part(i_a, v);
                    fence_proxy_async();
                    mbar_arrive(&s_lo);   // the first half of S_{c+1}^T is in place
                    if (has_row) store_part(i_b, v + QP);
                    fence_proxy_async();
                    mbar_arrive(&s_hi);   // and the second
                } else if (has_row && p.hT) {
#pragma unroll
                    for (int hp = 0; hp < 2; ++hp) {
                        const int i0 = hp ? i_b : i_a;
                        const uint32_t *vp = v + hp * QP;
                        if (vf) {   // value-major: row j of the state is contiguous
                            float *dst = p.hT + hbase + (size_t)j * D + i0;
#pragma unroll
                            for (int i = 0; i < QP; i += 4)
                                *reinterpret_cast<float4 *>(dst + i) =
                                    make_float4(__uint_as_float(vp[i]), __uint_as_float(vp[i + 1]),
                                                __uint_as_float(vp[i + 2]), __uint_as_float(vp[i + 3]));
                        } else {
#pragma unroll
                            for (int i = 0; i < QP; ++i)
                                p.hT[hbase + (size_t)(i0 + i) * D + j] = __uint_as_float(vp[i]);
                        }
                    }
                }
                if (has_row && !last && p.states) {
                    // the state the next chunk starts from, kept for the backward in bf16, the
                    // precision of the operand the walk itself carries (after the arrives:
                    // these stores stay off the walk's critical path)
                    __nv_bfloat16 *base = dump_at(REV ? t.nc - 2 - c : c + 1) + j;
#pragma unroll
                    for (int i = 0; i < QP; ++i) {
                        base[(size_t)(i_a + i) * D] = __float2bfloat16_rn(__uint_as_float(v[i]));
                        base[(size_t)(i_b + i) * D] = __float2bfloat16_rn(__uint_as_float(v[QP + i]));
                    }
                }
            }
        }
    } else if (warp < 14) {
        // ---------------- output epilogue, warps 10..13: O[t][j] from the same
        // accumulator, staged row-major [t][j] and written out as whole 16-byte rows.
        const int q = warp & 3;
        const bool has_row = (D == 128) || (lane < 16);
        const int j = (D == 128) ? 32 * q + lane : 16 * q + lane;
        const uint32_t lrow = (uint32_t)(32 * q) << 16;
        const int et = tid - 320;       // 0..127 over the output warps
        __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sO);
        constexpr int CPR = D / 8;      // 16-byte pieces per output row
        // Every output warp passes both named barriers of every chunk, failed or not (a
        // warp that left the loop early would leave the others waiting at the barrier);
        // after a failure the remaining chunks are skipped without waiting.  The reverse
        // walk writes its fp32 value gradients straight from the registers instead (token
        // by token, the warp's 32 value columns contiguous).
        int gc = 0;
        for (int r = 0; chain_task(p, chain, r, t); ++r) {
            for (int c = 0; c < t.nc; ++c, ++gc) {
                const int b = gc & 1;
                bool ok = !s_fail;
                if (ok && !mbar_wait(&d_full[b], (gc >> 1) & 1, kWaitNs)) {
                    s_fail = 1;
                    record_error(p.ws, 14);
                    ok = false;
                }
                uint32_t v[kC];
                if (ok) {
                    tc_fence_after();
                    const uint32_t dcol = tm + lrow + (uint32_t)(b * R);
                    if (!REV || p.dv_out) {
                        tmem_ld32(dcol + D, *reinterpret_cast<uint32_t(*)[32]>(v));
                        tmem_ld32(dcol + D + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                        tmem_ld_wait();
                    }
                    tc_fence_before();
                    mbar_arrive(&d_free[b]);
                }
                if (REV) {   // (dv_out may be nullptr: the value gradients are formed elsewhere)
                    const int cc = t.nc - 1 - c;
                    const int nv = ok ? min(kC, t.len - cc * kC) : 0;
                    if (has_row && p.dv_out)
                        for (int tt = 0; tt < nv; ++tt)
                            p.dv_out[((size_t)(t.start + (long)cc * kC + tt) * p.H + t.h) * D + j] =
                                __uint_as_float(v[tt]);
                    continue;
                }
                named_sync(1, 128);          // the previous chunk's rows have been written out
                if (ok && has_row)
#pragma unroll
                    for (int tt = 0; tt < kC; ++tt) stg[tt * D + j] = __float2bfloat16_rn(__uint_as_float(v[tt]));
                named_sync(1, 128);
                const int nv = (ok && p.o) ? min(kC, t.len - c * kC) : 0;
                __nv_bfloat16 *obase = p.o + ((size_t)(t.start + (long)c * kC) * p.H + t.h) * D;
#pragma unroll
                for (int k = et; k < kC * CPR; k += 128) {
                    const int tt = k / CPR, cc = k % CPR;
                    if (tt < nv)
                        *reinterpret_cast<uint4 *>(obase + (size_t)tt * p.H * D + cc * 8) =
                            *reinterpret_cast<const uint4 *>(stg + tt * D + cc * 8);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tm, Cf::TCOLS);
    }
}

// ---------------------------------------------------------------------------------
// tc_kernel -- CTAs [0, nch) take the chain role, the others hold the prep groups (two of
// 256 threads, or one of 512 for the per-channel decay).  The launch is cooperative: every
// chain is co-resident with the prep groups it waits for, and they with it.
// ---------------------------------------------------------------------------------
template <int D, bool GK, bool OPT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(const __grid_constant__ CUtensorMap map_q,
                                                           const __grid_constant__ CUtensorMap map_k,
                                                           const __grid_constant__ CUtensorMap map_v,
                                                           const __grid_constant__ CUtensorMap map_E,
                                                           const __grid_constant__ CUtensorMap map_Ew,
                                                           TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    if ((int)blockIdx.x < p.nch) {
        chain_body<D, OPT>(&map_E, &map_v, p, sm, (int)blockIdx.x);
        return;
    }
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, grp = tid >> 8;
    if constexpr (GK) {   // one prep group of all 512 threads per CTA
        if (tid == 0) {
            PrepCtrl *ctl = reinterpret_cast<PrepCtrl *>(sm + GkSmem<D>::CTRL);
            mbar_init(&ctl->bar_mma, 1);
            fence_mbar_init();
            ctl->fail = 0;
        }
        if (tid < 32) {
            tmem_alloc(&tmem_base, 256);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        prep_group_gk<D, OPT>(&map_Ew, p, sm, tmem_base, tid, 1);
        tc_fence_before();
        __syncthreads();
        if (tid < 32) {
            __syncwarp();
            tmem_dealloc(tmem_base, 256);
        }
        return;
    }
    uint8_t *gsm = sm + grp * PrepSmem<D>::GROUP;
    if ((tid & (kGroupThreads - 1)) == 0) {
        PrepCtrl *ctl = reinterpret_cast<PrepCtrl *>(gsm + PrepSmem<D>::CTRL);
        mbar_init(&ctl->bar_mma, 1);
        fence_mbar_init();
        ctl->fail = 0;
    }
    if (tid < 32) {   // 256 columns for each group
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const long ngroups = (long)((int)gridDim.x - p.nch) * 2;
    const bool stagger = prep_items(p) >= 16 * ngroups;   // long runs only: the offset costs a start-up delay
    prep_group<D, OPT>(&map_q, &map_k, &map_E, p, gsm, tmem_base + (uint32_t)(grp * 256),
                  tid & (kGroupThreads - 1), 1 + grp, stagger);
    tc_fence_before();
    __syncthreads();
    if (tid < 32) {
        __syncwarp();
        tmem_dealloc(tmem_base, 512);
    }
}

// Failure-detection probe: the two bounded waits of the kernels above, run against events
// that never happen (an mbarrier phase nobody arrives on, a flag nobody releases) with a
// short limit; each time-out is recorded in the workspace header like a kernel's would be.
__global__ void timeout_probe_kernel(WsHeader *ws, const uint32_t *never, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, limit_ns)) record_error(ws, 90);
        if (!wait_flag_acquire(never, 1u, limit_ns)) record_error(ws, 91);
    }
}

// Packed sequences: the order of the tasks and the columns of the rounds.
//   order[rank]  = the sequence of that rank by decreasing chunk count (ties: lower index
//                  first); the identity for more than kSortMax sequences
//   round_base[r] = sum over rounds r' < r of the largest chunk count among the round's
//                  sequences; round r holds tasks [r nch, (r + 1) nch), task = rank H + head.
// One CTA.
constexpr int kSortMax = 2048;
__global__ void varlen_schedule_kernel(const int *cu, int N, int H, int nch, int rounds, int *order,
                                       int *round_base) {
    __shared__ int snc[kSortMax];
    const int tid = threadIdx.x;
    const bool sort = N <= kSortMax;
    auto nc_of = [&](int n) { return (cu[n + 1] - cu[n] + kC - 1) / kC; };
    if (sort)
        for (int n = tid; n < N; n += blockDim.x) snc[n] = nc_of(n);
    __syncthreads();
    for (int n = tid; n < N; n += blockDim.x) {
        if (!sort) {
            order[n] = n;
            continue;
        }
        const int mine = snc[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int o = snc[m];
            rank += (o > mine) || (o == mine && m < n);
        }
        order[rank] = n;
    }
    __syncthreads();
    if (tid == 0) {   // rounds <= N * H; sorted: the round's first sequence is its longest
        int acc = 0;
        for (int r = 0; r < rounds; ++r) {
            round_base[r] = acc;
            const int first = (int)(((long)r * nch) / H);   // ranks of the round's tasks
            const int last = (int)(min((long)(r + 1) * nch, (long)N * H) - 1) / H;
            int m = 0;
            for (int k = first; k <= (sort ? first : last); ++k) m = max(m, nc_of(order[k]));
            acc += m;
        }
        round_base[rounds] = acc;
    }
}

bool map_tokens(CUtensorMap *m, const void *base, long rows, int H, int D) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)H, (uint64_t)rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)H * D * 2};
    const uint32_t box[3] = {64u, 1u, 64u};
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, true);
}

bool map_E(CUtensorMap *m, const void *base, long slots, int R) {
    const uint64_t dims[3] = {(uint64_t)R, (uint64_t)R, (uint64_t)slots};
    const uint64_t strides[2] = {(uint64_t)R * 2, (uint64_t)R * R * 2};
    const uint32_t box[3] = {64u, (uint32_t)R, 1u};
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, true);
}
// E_c written in 16-row x 32-column boxes from 64-byte-swizzled staging tiles
bool map_E_tiles(CUtensorMap *m, const void *base, long slots, int R) {
    const uint64_t dims[3] = {(uint64_t)R, (uint64_t)R, (uint64_t)slots};
    const uint64_t strides[2] = {(uint64_t)R * 2, (uint64_t)R * R * 2};
    const uint32_t box[3] = {32u, 16u, 1u};
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Chains for `ntask` tasks on `nsm` SMs: at most a quarter of the SMs (the prep is the
// larger share of the work) and kMaxChains, balanced so that every round but the last is
// full and the last nearly so.
int chains_for(long ntask, int nsm) {
    long nch = std::min<long>(std::min<long>(ntask, nsm / 4), kMaxChains);
    if (nch < 1) nch = 1;
    const long rounds = (ntask + nch - 1) / nch;
    return (int)((ntask + rounds - 1) / rounds);
}

// Scratch layout after the workspace header (chains <= nch_max):
//   [order: nseq ints][round_base: ntask + 1 ints]   packed sequences only
//   [flags: nch_max * kRing][consumed: nch_max][next item: 1]   uint32, each counter on its own 128-byte line
//   [E_c rings: nch_max * kRing * (D + 64)^2 bf16]
struct ScratchLayout {
    size_t order, round_base, flags, consumed, E, total;
};
// keep_nc > 0: the maps of every chunk are kept for a reverse walk (equal-length batches of
// keep_nc chunks): each chain's ring holds all of its columns, rounds x keep_nc.
ScratchLayout scratch_layout(int nseq, int H, int d, bool varlen, int keep_nc = 0) {
    const long ntask = (long)nseq * H;
    const long nch_max = std::max<long>(1, std::min<long>(ntask, kMaxChains));
    const size_t R = (size_t)d + 64;
    // slots: chains x ring; when keeping, chains x rounds x keep_nc <= (ntask + chains) x keep_nc
    const size_t slots = keep_nc > 0 ? (size_t)(ntask + nch_max) * keep_nc : (size_t)nch_max * kRing;
    ScratchLayout L{};
    size_t off = 0;
    L.order = off;
    if (varlen) off += align256((size_t)nseq * 4);
    L.round_base = off;
    if (varlen) off += align256((size_t)(ntask + 1) * 4);
    L.flags = off;
    off += align256(slots * 4);
    L.consumed = off;
    off += align256((size_t)(nch_max + 1) * kCounterStride * 4);
    L.E = off;
    off += slots * R * R * 2;
    L.total = off;
    return L;
}

// What a forward launch that kept its maps leaves for the reverse walk.
struct TcPlan {
    int nch, ring, rounds;
    __nv_bfloat16 *E;
};

// OPT: the kda_options paths, compiled out of the plain instantiations
// states: or nullptr, the state at every chunk start (bf16); keep: or nullptr, every chunk's
// map stays in the scratch and the plan is returned (equal-length batches only).
template <int D, bool GK, bool OPT>
cudaError_t run_tc(const SeqBatch &a, long total_rows, cudaStream_t st, __nv_bfloat16 *states = nullptr,
                   TcPlan *keep = nullptr) {
    constexpr int R = D + 64;
    using Cf = ChainCfg<D>;
    TcParams p{};
    p.nseq = a.nseq; p.H = a.H; p.T = a.T; p.use_l2 = a.use_l2; p.scale = a.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.nc_equal = (a.T + kC - 1) / kC;
    p.beta = a.beta; p.decay = GK ? nullptr : a.decay; p.h0 = a.h0; p.hT = a.hT;
    p.gk = GK ? a.gk : nullptr;
    p.decayed_read = a.decayed_read;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias; p.beta_sig = a.beta_sig; p.neg_eig = a.neg_eig;
    p.G = a.G > 1 ? a.G : 1;
    p.v_first = a.v_first;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k = static_cast<const __nv_bfloat16 *>(a.k);
    p.rows = total_rows;
    p.o = static_cast<__nv_bfloat16 *>(a.o);
    p.ws = a.ws;
    p.ntask = a.nseq * a.H;
    const bool varlen = a.cu_seqlens != nullptr;
    if (keep && varlen) return cudaErrorInvalidValue;
    p.states = states;
    const ScratchLayout L = scratch_layout(a.nseq, a.H, D, varlen, keep ? p.nc_equal : 0);
    if (L.total > a.ws_body_bytes) return cudaErrorInvalidValue;
    uint8_t *body = static_cast<uint8_t *>(a.ws_body);
    p.order = varlen ? reinterpret_cast<const int *>(body + L.order) : nullptr;
    p.round_base = varlen ? reinterpret_cast<const int *>(body + L.round_base) : nullptr;
    p.flags = reinterpret_cast<uint32_t *>(body + L.flags);
    p.consumed = reinterpret_cast<uint32_t *>(body + L.consumed);
    p.next_item = p.consumed + std::max<long>(1, std::min<long>(p.ntask, kMaxChains)) * kCounterStride;
    p.E = reinterpret_cast<__nv_bfloat16 *>(body + L.E);

    int dev = 0, nsm = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int prep_smem = GK ? GkSmem<D>::BYTES + 1024 : 2 * PrepSmem<D>::GROUP + 1024;
    const int one_smem = std::max(prep_smem, Cf::SMEM);
    e = cudaFuncSetAttribute(tc_kernel<D, GK, OPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, one_smem);
    if (e != cudaSuccess) return e;

    // One cooperative launch: chains and prep groups co-resident.  If fewer SMs can take a
    // block than the device reports (a partitioned GPU), the grid shrinks and the chains
    // with it (the kernel is persistent: any grid with a prep CTA works).
    for (int grid = nsm; grid >= 2; grid -= std::max(1, grid / 8)) {
        p.nch = chains_for(p.ntask, grid);
        p.rounds = (p.ntask + p.nch - 1) / p.nch;
        p.ring = keep ? p.rounds * p.nc_equal : kRing;
        const long cols = varlen ? (long)p.rounds * ((a.T + kC - 1) / kC) : (long)p.rounds * p.nc_equal;
        if (cols * p.nch >= (1L << 31)) return cudaErrorInvalidValue;   // 32-bit item indexing
        const size_t fbytes = reinterpret_cast<uint8_t *>(p.next_item + 1) - (body + L.flags);
        if ((e = cudaMemsetAsync(body + L.flags, 0, fbytes, st)) != cudaSuccess) return e;
        if (varlen) {
            varlen_schedule_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.nseq, a.H, p.nch, p.rounds,
                                                       reinterpret_cast<int *>(body + L.order),
                                                       reinterpret_cast<int *>(body + L.round_base));
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        CUtensorMap mq, mk, mv, me, mew;
        const long slots = (long)p.nch * p.ring;
        if (!map_tokens(&mq, a.q, total_rows, a.H / p.G, D) || !map_tokens(&mk, a.k, total_rows, a.H / p.G, D) ||
            !map_tokens(&mv, a.v, total_rows, a.H, D) || !map_E(&me, p.E, slots, R) ||
            !map_E_tiles(&mew, p.E, slots, R))
            return cudaErrorInvalidValue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = (size_t)one_smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc_kernel<D, GK, OPT>, mq, mk, mv, me, mew, p);
        if (e == cudaSuccess && keep) *keep = TcPlan{p.nch, p.ring, p.rounds, p.E};
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        (void)cudaGetLastError();
    }
    return cudaErrorCooperativeLaunchTooLarge;
}

// The reverse walk over the maps a forward launch kept (plan): one chain CTA per task
// slot of the forward, chunks last to first; d_o streamed like v, dhT in, dh0 out (either
// may be nullptr: zeros in, not written), dv and the incoming state gradient of every chunk
// (dstates) out.
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) rev_chain_kernel(const __grid_constant__ CUtensorMap map_E,
                                                                  const __grid_constant__ CUtensorMap map_do,
                                                                  TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    chain_body<D, false, true>(&map_E, &map_do, p, align1024(smem_raw), (int)blockIdx.x);
}

template <int D>
cudaError_t run_rev(const SeqBatch &a, const TcPlan &plan, const void *d_o, const float *dhT, float *dh0,
                    float *dv, __nv_bfloat16 *dstates, cudaStream_t st) {
    constexpr int R = D + 64;
    using Cf = ChainCfg<D>;
    TcParams p{};
    p.nseq = a.nseq; p.H = a.H; p.T = a.T;
    p.nc_equal = (a.T + kC - 1) / kC;
    p.h0 = dhT; p.hT = dh0;
    p.rows = (long)a.nseq * a.T;
    p.ws = a.ws;
    p.ntask = a.nseq * a.H;
    p.nch = plan.nch; p.rounds = plan.rounds; p.ring = plan.ring;
    p.E = plan.E;
    p.states = dstates;
    p.dv_out = dv;
    CUtensorMap me, mdo;
    if (!map_E(&me, p.E, (long)p.nch * p.ring, R) || !map_tokens(&mdo, d_o, p.rows, a.H, D))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(rev_chain_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    rev_chain_kernel<D><<<(unsigned)p.nch, kTcThreads, Cf::SMEM, st>>>(me, mdo, p);
    return cudaGetLastError();
}

}  // namespace

bool chunk_tc_supported(int dk, int dv, int chunk, DType dt) {
    return dt == DType::BF16 && dk == dv && (dk == 64 || dk == 128) && chunk == kC;
}

// Scratch bytes after the workspace header: the rings of the chains (at most kMaxChains,
// whatever the sequence length) and, for packed sequences, the schedule tables.
size_t chunk_tc_scratch_bytes(int nseq, int H, int d, bool varlen) {
    return scratch_layout(nseq, H, d, varlen).total;
}

cudaError_t launch_timeout_probe(WsHeader *ws, uint64_t limit_ns, cudaStream_t st) {
    uint32_t *never = &ws->probe;   // zeroed here, released by nobody
    cudaError_t e = cudaMemsetAsync(never, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    timeout_probe_kernel<<<1, 32, 0, st>>>(ws, never, limit_ns);
    return cudaGetLastError();
}

size_t chunk_tc_keep_bytes(int B, int H, int T, int d) {
    return scratch_layout(B, H, d, false, (T + kC - 1) / kC).total;
}

cudaError_t launch_chunk_tc_walks(const SeqBatch &a, const void *d_o, const float *dhT, float *dh0, float *dv,
                                  __nv_bfloat16 *fstates, __nv_bfloat16 *bstates, cudaStream_t st) {
    if ((long)a.nseq * a.T >= (1L << 31) || a.cu_seqlens) return cudaErrorInvalidValue;
    // the per-channel prep takes the decayed read at run time; the scalar one compiles it in
    const bool opt = a.decayed_read != 0 && !a.per_channel;
    const long rows = (long)a.nseq * a.T;
    TcPlan plan{};
    cudaError_t e;
    if (a.dk == 128) {
        e = a.per_channel ? run_tc<128, true, false>(a, rows, st, fstates, &plan)
            : opt         ? run_tc<128, false, true>(a, rows, st, fstates, &plan)
                          : run_tc<128, false, false>(a, rows, st, fstates, &plan);
        return e != cudaSuccess ? e : run_rev<128>(a, plan, d_o, dhT, dh0, dv, bstates, st);
    }
    if (a.dk == 64) {
        e = a.per_channel ? run_tc<64, true, false>(a, rows, st, fstates, &plan)
            : opt         ? run_tc<64, false, true>(a, rows, st, fstates, &plan)
                          : run_tc<64, false, false>(a, rows, st, fstates, &plan);
        return e != cudaSuccess ? e : run_rev<64>(a, plan, d_o, dhT, dh0, dv, bstates, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_tc(const SeqBatch &a, long total_rows, cudaStream_t st) {
    if (total_rows >= (1L << 31)) return cudaErrorInvalidValue;   // 32-bit row indexing
    if (a.per_channel) {   // the decayed read is a runtime choice of the per-channel prep
        const bool gopt = a.A_log || a.beta_sig || a.G > 1 || a.v_first;
        if (a.dk == 128)
            return gopt ? run_tc<128, true, true>(a, total_rows, st) : run_tc<128, true, false>(a, total_rows, st);
        if (a.dk == 64)
            return gopt ? run_tc<64, true, true>(a, total_rows, st) : run_tc<64, true, false>(a, total_rows, st);
        return cudaErrorInvalidValue;
    }
    const bool opt = a.decayed_read || a.A_log || a.beta_sig || a.G > 1 || a.v_first;
    if (a.dk == 128)
        return opt ? run_tc<128, false, true>(a, total_rows, st) : run_tc<128, false, false>(a, total_rows, st);
    if (a.dk == 64)
        return opt ? run_tc<64, false, true>(a, total_rows, st) : run_tc<64, false, false>(a, total_rows, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
