// kda_api.cu -- the extern "C" entry points of libkda: argument validation,
// workspace carving, TMA descriptor encoding, and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "kda_internal.h"

namespace {

using kda::kHeadDim;

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

// Device must be sm_103 (the kernels are built for sm_103a only).
kda_status check_device() {
    static int support[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices && support[dev] != 0) return support[dev] == 1 ? KDA_OK : KDA_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < kMaxDevices) support[dev] = ok ? 1 : 2;
    return ok ? KDA_OK : KDA_ERR_UNSUPPORTED;
}

}  // namespace

namespace kda {
kda_status device_check() { return check_device(); }
}  // namespace kda

namespace {

int sm_count() {
    static int count[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (count[dev] == 0) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) count[dev] = c;
    }
    return count[dev];
}

// Piecewise schedule of the two-pass prefill.  When the scan takes at most half
// of the GPU's SMs (few sequences), the scan runs in pieces of 48 or more
// chunks per sequence (at most 32 pieces) and pass 1 runs ahead of it, all on
// the caller's stream: a first pass-1 launch prepares a lead of chunks on the
// whole GPU; then each scan piece is followed by the next pass-1 share,
// launched as a programmatic dependent of that piece, so that it starts once
// every CTA of the piece is running and takes only the SMs the scan leaves
// idle (pass 2 then reads images written moments earlier, still in L2).  Each
// scan piece is an ordinary launch: it starts after everything before it on
// the stream, the previous piece (whose S_final carries the state) and the
// pass-1 shares included.  Each piece boundary costs a few microseconds
// (launch, state carry, first copies), which bounds the piece count.
constexpr int64_t kScanPieceChunks = 48;  // smallest scan piece (chunks per sequence); each piece costs a few us
constexpr int64_t kMaxScanPieces = 32;     // longer sequences get longer pieces
// lead of pass 1, as a fraction of the chunks scanned after piece 0 (A/B of 0.1 / 0.05 / 0.02 / 0: 8k
// 322 / 317 / 319 / 321 us, 1M tokens 28.15 / 27.46 / 27.30 / 27.32 ms, two 32k sequences 2.10 / 2.11 /
// 2.11 / 2.11 ms)
constexpr double kPrepLag = 0.05;
// the same with the fused prologue (a slower pass 1): A/B of 0.2 / 0.1 / 0.05, 8k with the prologue
// 337.1 / 333.8 / 339.2 us, with every fusion 372.1 / 369.3 / 375.8 us
constexpr double kPrepLagPrologue = 0.1;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a [T][H][inner] tensor, box = {box_inner, 1, box_rows}.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t inner, uint64_t H,
              uint64_t T, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, H, T > 0 ? T : 1};
    const cuuint64_t strides[2] = {inner * esize, H * inner * esize};
    const cuuint32_t box[3] = {box_inner, 1, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t esize_of(kda_dtype t) { return t == KDA_DTYPE_F32 ? 4 : 2; }

// Workspace layouts.  Two-pass path: [schedule][chunk table][bf16 q,k,v if
// fp32 inputs][per-(chunk, head) operand images].  Single-pass path:
// [schedule][bf16 q,k,v if fp32 inputs].
struct WsLayout {
    size_t table = 0, copies = 0, blobs = 0, carry = 0, total = 0;
};
size_t copies_bytes(kda_dtype t, int64_t T, int32_t H) {
    if (t != KDA_DTYPE_F32) return 0;
    const size_t n = static_cast<size_t>(T) * H * kHeadDim;
    return 3 * round_up(n * 2, kAlign);
}
int64_t max_chunks(int32_t N, int64_t T) { return (T + kda::kChunk - 1) / kda::kChunk + N; }
WsLayout split_layout(kda_dtype t, int32_t N, int64_t T, int32_t H) {
    WsLayout w;
    w.table = round_up(static_cast<size_t>(N > 0 ? N : 1) * 4, kAlign);
    w.copies = w.table + round_up(static_cast<size_t>(N + 2) * 4, kAlign);  // chunk table
    w.blobs = w.copies + copies_bytes(t, T, H);
    // the state carried between scan pieces when the caller asks for no S_final
    w.carry = round_up(w.blobs + static_cast<size_t>(max_chunks(N, T)) * H * kda::kPrefillBlobBytes, kAlign);
    w.total = w.carry + static_cast<size_t>(N) * H * kHeadDim * kHeadDim * 4;
    return w;
}
WsLayout fused_layout(kda_dtype t, int32_t N, int64_t T, int32_t H) {
    WsLayout w;
    w.copies = round_up(static_cast<size_t>(N > 0 ? N : 1) * 4, kAlign);
    w.total = w.copies + copies_bytes(t, T, H);
    return w;
}
bool ws_args_ok(kda_dtype t, int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv);

bool sizes_ok(int64_t a, int64_t b, int64_t c, int64_t d) {  // product fits comfortably in int64
    const double prod = static_cast<double>(a) * static_cast<double>(b) * static_cast<double>(c) *
                        static_cast<double>(d);
    return prod < 4.0e18;
}

bool ws_args_ok(kda_dtype t, int32_t N, int64_t T, int32_t H, int32_t dk, int32_t dv) {
    if (N < 0 || T < 0 || H <= 0 || dk != kHeadDim || dv != kHeadDim) return false;
    if (t != KDA_DTYPE_BF16 && t != KDA_DTYPE_F32) return false;
    return sizes_ok(T + N + 1, H, kda::kPrefillBlobBytes, 1) && sizes_ok(T, H, kHeadDim, 4);
}

}  // namespace

extern "C" {

int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    }
    return "KDA_ERR_UNKNOWN";
}

size_t kda_prefill_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                   int32_t dk, int32_t dv) {
    if (!ws_args_ok(qkv_dtype, num_seqs, total_tokens, H, dk, dv)) return 0;
    return split_layout(qkv_dtype, num_seqs, total_tokens, H).total;
}

size_t kda_prefill_min_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                       int32_t dk, int32_t dv) {
    if (!ws_args_ok(qkv_dtype, num_seqs, total_tokens, H, dk, dv)) return 0;
    return fused_layout(qkv_dtype, num_seqs, total_tokens, H).total;
}

}  // extern "C"

namespace {

// Fusion options: validated copy (flags 0 when `f` is NULL).  Returns false on
// unknown flags, a negative eps, a missing / misaligned out_gate or weight.
// `rows`: whether the call has any (token, head) rows; without them out_gate, like every other
// zero-size array, may be NULL.
bool fusion_ok(const kda_fusion* f, kda::DecodeFusion& out, bool rows) {
    out = kda::DecodeFusion();
    if (!f) return true;
    constexpr uint32_t known = KDA_FUSE_L2NORM_QK | KDA_FUSE_BETA_SIGMOID | KDA_FUSE_OUT_GATE;
    if (f->flags & ~known) return false;
    if (!(f->l2_eps >= 0.f) || !(f->rms_eps >= 0.f)) return false;
    if ((f->flags & KDA_FUSE_OUT_GATE) && ((rows && !f->out_gate) || !aligned(f->out_gate, 16))) return false;
    if (f->rms_weight && !aligned(f->rms_weight, 4)) return false;
    out.flags = f->flags;
    out.l2_eps = f->l2_eps;
    out.rms_eps = f->rms_eps;
    out.rms_weight = f->rms_weight;
    out.out_gate = f->out_gate;
    return true;
}

struct Snapshots {
    const int32_t* seq = nullptr;
    const int32_t* pos = nullptr;
    int32_t count = 0;
    float* S = nullptr;
};

kda_status prefill_impl(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                        const float* beta, const float* S0, const int32_t* cu_seqlens, int32_t num_seqs,
                        int64_t total_tokens, int32_t H, int32_t dk, int32_t dv, void* o, float* S_final,
                        const Snapshots& snap, const kda_fusion* fusion, void* workspace, size_t workspace_bytes,
                        int32_t* device_status, kda_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    kda::DecodeFusion fz;
    if (!fusion_ok(fusion, fz, total_tokens > 0)) return KDA_ERR_INVALID_ARG;
    if (qkv_dtype != KDA_DTYPE_BF16 && qkv_dtype != KDA_DTYPE_F32) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || total_tokens > INT32_MAX - 64) return KDA_ERR_INVALID_ARG;
    if (dk != kHeadDim || dv != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (!sizes_ok(total_tokens, H, kHeadDim, 4) || !sizes_ok(num_seqs, H, kHeadDim, kHeadDim * 4))
        return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !workspace) return KDA_ERR_INVALID_ARG;
    const bool have_tokens = total_tokens > 0;
    if (have_tokens && (!q || !k || !v || !log_alpha || !beta || !o)) return KDA_ERR_INVALID_ARG;
    const size_t es = esize_of(qkv_dtype);
    const size_t nqk = static_cast<size_t>(total_tokens) * H * kHeadDim;
    const size_t nst = static_cast<size_t>(num_seqs) * H * kHeadDim * kHeadDim;
    if (have_tokens && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, 16) ||
                        !aligned(o, 16) || !aligned(beta, 4)))
        return KDA_ERR_INVALID_ARG;
    if ((S0 && !aligned(S0, 16)) || (S_final && !aligned(S_final, 16)) || !aligned(workspace, kAlign) ||
        !aligned(cu_seqlens, 4) || (device_status && !aligned(device_status, 4)))
        return KDA_ERR_INVALID_ARG;
    // Path by workspace size: the two-pass path when the workspace holds the
    // per-(chunk, head) operand images, else the single-pass path.
    if (kda_prefill_workspace_bytes(qkv_dtype, num_seqs, total_tokens, H, dk, dv) == 0) return KDA_ERR_INVALID_ARG;
    const WsLayout two = split_layout(qkv_dtype, num_seqs, total_tokens, H);
    const WsLayout one = fused_layout(qkv_dtype, num_seqs, total_tokens, H);
    const bool two_pass = workspace_bytes >= two.total;
    if (!two_pass && workspace_bytes < one.total) return KDA_ERR_WORKSPACE;
    const WsLayout& lay = two_pass ? two : one;
    const size_t need = lay.total;
    if (snap.count < 0) return KDA_ERR_INVALID_ARG;
    if (snap.count > 0) {
        if (!snap.seq || !snap.pos || !snap.S || !aligned(snap.seq, 4) || !aligned(snap.pos, 4) || !aligned(snap.S, 16))
            return KDA_ERR_INVALID_ARG;
        if (!sizes_ok(snap.count, H, kHeadDim, kHeadDim * 4)) return KDA_ERR_INVALID_ARG;
        if (!two_pass) return KDA_ERR_WORKSPACE;
    }
    if (fz.flags && !two_pass) return KDA_ERR_WORKSPACE;

    // Overlap rules: outputs overlap nothing (S_final may equal S0 exactly).
    const Range r_o = range_of(o, nqk * es), r_sf = range_of(S_final, S_final ? nst * 4 : 0);
    const Range r_ws = range_of(workspace, need);
    const Range inputs[] = {range_of(q, nqk * es),          range_of(k, nqk * es),
                            range_of(v, nqk * es),          range_of(log_alpha, nqk * 4),
                            range_of(beta, static_cast<size_t>(total_tokens) * H * 4),
                            range_of(cu_seqlens, static_cast<size_t>(num_seqs + 1) * 4),
                            range_of(device_status, device_status ? 4 : 0)};
    const Range r_s0 = range_of(S0, S0 ? nst * 4 : 0);
    for (const Range& in : inputs) {
        if (have_tokens && overlap(r_o, in)) return KDA_ERR_INVALID_ARG;
        if (overlap(r_sf, in) || overlap(r_ws, in)) return KDA_ERR_INVALID_ARG;
    }
    if (have_tokens && (overlap(r_o, r_sf) || overlap(r_o, r_ws) || overlap(r_o, r_s0))) return KDA_ERR_INVALID_ARG;
    if (overlap(r_sf, r_ws) || overlap(r_s0, r_ws)) return KDA_ERR_INVALID_ARG;
    if (S0 && S_final && S0 != S_final && overlap(r_sf, r_s0)) return KDA_ERR_INVALID_ARG;
    if (fz.flags & KDA_FUSE_OUT_GATE) {  // out_gate is read while o is written
        const Range r_g = range_of(fz.out_gate, nqk * es);
        if (have_tokens && overlap(r_g, r_o)) return KDA_ERR_INVALID_ARG;
        if (overlap(r_g, r_sf) || overlap(r_g, r_ws)) return KDA_ERR_INVALID_ARG;
    }
    if (snap.count > 0) {  // S_snap is an output: it overlaps nothing
        const Range r_ss = range_of(snap.S, static_cast<size_t>(snap.count) * H * kHeadDim * kHeadDim * 4);
        const Range r_sq = range_of(snap.seq, static_cast<size_t>(snap.count) * 4);
        const Range r_sp = range_of(snap.pos, static_cast<size_t>(snap.count) * 4);
        for (const Range& in : inputs)
            if (overlap(r_ss, in)) return KDA_ERR_INVALID_ARG;
        if (overlap(r_ss, r_sq) || overlap(r_ss, r_sp) || overlap(r_ss, r_ws) || overlap(r_ss, r_s0) ||
            overlap(r_ss, r_sf) || (have_tokens && overlap(r_ss, r_o)))
            return KDA_ERR_INVALID_ARG;
    }

    const kda_status dev = check_device();
    if (dev != KDA_OK) return dev;
    if (!encode_fn()) return KDA_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* order = reinterpret_cast<int32_t*>(ws);
    size_t off = lay.copies;
    const void* qb = q;
    const void* kb = k;
    const void* vb = v;
    if (qkv_dtype == KDA_DTYPE_F32 && have_tokens) {
        void* qc = ws + off;
        off += round_up(nqk * 2, kAlign);
        void* kc = ws + off;
        off += round_up(nqk * 2, kAlign);
        void* vc = ws + off;
        if (kda::launch_to_bf16(static_cast<const float*>(q), qc, nqk, stream) != cudaSuccess ||
            kda::launch_to_bf16(static_cast<const float*>(k), kc, nqk, stream) != cudaSuccess ||
            kda::launch_to_bf16(static_cast<const float*>(v), vc, nqk, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        qb = qc;
        kb = kc;
        vb = vc;
    }
    // TMA maps need a valid base even when there are no tokens (never dereferenced then).
    const void* dummy = workspace;
    CUtensorMap tm_q, tm_k, tm_v, tm_la;
    const uint64_t T = static_cast<uint64_t>(total_tokens), Hh = static_cast<uint64_t>(H);
    // q, k, v: 64-channel boxes in the 128B-swizzled layout the tensor cores read
    if (!make_map(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, have_tokens ? qb : dummy, kHeadDim, Hh, T, 64,
                  kda::kChunk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, have_tokens ? kb : dummy, kHeadDim, Hh, T, 64,
                  kda::kChunk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, have_tokens ? vb : dummy, kHeadDim, Hh, T, 64,
                  kda::kChunk, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_la, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, have_tokens ? static_cast<const void*>(log_alpha) : dummy,
                  kHeadDim, Hh, T, kHeadDim, kda::kChunk, CU_TENSOR_MAP_SWIZZLE_NONE))
        return KDA_ERR_CUDA;
    // the snapshots as [entries x H x 128 rows][128] fp32: the scan stores 32 x 32 blocks, 128B-swizzled
    CUtensorMap tm_snap;
    const bool have_snaps = snap.count > 0;
    const uint64_t snap_rows =
        have_snaps ? std::min<uint64_t>(static_cast<uint64_t>(snap.count) * Hh * kHeadDim, kda::kSnapMapRows) : kHeadDim;
    if (!make_map(&tm_snap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, have_snaps ? static_cast<const void*>(snap.S) : dummy,
                  kHeadDim, 1, snap_rows, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return KDA_ERR_CUDA;
    const bool og = (fz.flags & KDA_FUSE_OUT_GATE) != 0;

    // the longest-first order of the sequences; one sequence in the two-pass path needs none (its chunk
    // table kernel checks cu_seqlens as the schedule kernel does)
    const bool need_order = !two_pass || num_seqs > 1;
    if (need_order &&
        kda::launch_schedule(cu_seqlens, num_seqs, total_tokens, order, device_status, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    kda::PrefillArgs a;
    a.log_alpha = log_alpha;
    a.beta = beta;
    a.S0 = S0;
    a.cu_seqlens = cu_seqlens;
    a.order = need_order ? order : nullptr;
    a.chunk_off = two_pass ? reinterpret_cast<const int32_t*>(ws + two.table) : nullptr;
    a.blobs = two_pass ? ws + two.blobs : nullptr;
    a.blob_units = two_pass ? static_cast<int64_t>(max_chunks(num_seqs, total_tokens)) * H : 0;
    a.o = o;
    a.S_final = S_final;
    a.device_status = device_status;
    a.snap_seq = snap.seq;
    a.snap_pos = snap.pos;
    a.num_snaps = snap.count;
    a.S_snap = snap.S;
    a.l2_eps = fz.l2_eps;
    a.total_tokens = total_tokens;
    a.num_seqs = num_seqs;
    a.H = H;
    const bool out_f32 = qkv_dtype == KDA_DTYPE_F32;
    // pass 1 applies the prologue; the output gate runs after the scan, in place on o (one pass over o
    // and the gate: cheaper than exchanging row sums between the two dv slices inside the scan)
    a.fuse_flags = fz.flags & ~KDA_FUSE_OUT_GATE;
    auto out_gate = [&](bool ok) {
        if (!ok) return KDA_ERR_CUDA;
        if (og && kda::launch_out_gate(out_f32, o, fz.out_gate, fz.rms_weight, fz.rms_eps, total_tokens * H,
                                       stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        return KDA_OK;
    };
    if (two_pass) {
        if (kda::launch_chunk_table(cu_seqlens, num_seqs, total_tokens, reinterpret_cast<int32_t*>(ws + two.table),
                                    device_status, snap.seq, snap.pos, snap.count, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        // chunks of the longest possible sequence bound the pieces
        const int64_t seq_chunks = (total_tokens + kda::kChunk - 1) / kda::kChunk;
        // piece count from the smallest piece, then equal pieces (128 chunks: 43, 43, 42)
        const int64_t sq0 = std::max<int64_t>(kScanPieceChunks, (seq_chunks + kMaxScanPieces - 1) / kMaxScanPieces);
        const int64_t sq = (seq_chunks + (seq_chunks + sq0 - 1) / sq0 - 1) / ((seq_chunks + sq0 - 1) / sq0);
        const int64_t pieces = (seq_chunks + sq - 1) / sq;
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        // (a scan on more than half the SMs leaves pass 1 too few beside it: A/B, one prep + one scan
        // instead, 2 x 8192 tokens x 32 heads 559 -> 497 us, 4 x 16k x 16 heads 1267 -> 940 us, 3 x 32k x 16
        // heads 1779 -> 1552 us; two sequences of 32k + 20k tokens x 24 heads 1389 -> 1409 us)
        const bool piecewise = pieces > 1 && 2 * (static_cast<int64_t>(num_seqs) * H * 2) <= sm_count() &&
                               cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone;
        if (!piecewise)
            return out_gate(kda::launch_prefill_split(tm_q, tm_k, tm_v, tm_snap, a, max_chunks(num_seqs, total_tokens), out_f32,
                                                      stream) == cudaSuccess);
        // Scan piece j covers chunks [j sq, (j+1) sq).  Pass 1's first launch prepares a lead of L0
        // chunks; its launch j (j >= 1) prepares the next share of the rest beside scan piece j-1.  L0
        // makes up for pass 1 being slower on the SMs the scan leaves than the scan is per chunk.
        const int64_t lead = std::min<int64_t>(
            seq_chunks, sq + static_cast<int64_t>((a.fuse_flags ? kPrepLagPrologue : kPrepLag) *
                                                      static_cast<double>(sq * (pieces - 1)) + 0.999));
        const int64_t share = (seq_chunks - lead + pieces - 2) / (pieces - 1);
        if (!S_final) a.S_final = reinterpret_cast<float*>(ws + two.carry);  // the pieces' state carry
        bool ok = true;
        int64_t prepared = 0;  // chunks [0, prepared) of every sequence have their images (or are queued)
        for (int64_t j = 0; j < pieces && ok; ++j) {
            const int64_t scan_end = std::min(seq_chunks, (j + 1) * sq);
            int64_t prep_end = j == 0 ? lead : std::min(seq_chunks, lead + j * share);
            prep_end = std::max(prep_end, scan_end);
            if (prep_end > prepared) {
                a.piece_begin = static_cast<int32_t>(prepared);
                a.piece_len = static_cast<int32_t>(prep_end - prepared);
                ok = kda::launch_chunk_prep(tm_q, tm_k, a, static_cast<int64_t>(num_seqs) * a.piece_len, stream,
                                            j > 0) == cudaSuccess;
                prepared = prep_end;
            }
            a.piece_begin = static_cast<int32_t>(j * sq);
            a.piece_len = static_cast<int32_t>(scan_end - j * sq);
            ok = ok && kda::launch_chunk_scan(tm_v, tm_snap, a, out_f32, stream) == cudaSuccess;
        }
        return out_gate(ok);
    } else if (kda::launch_prefill_fused(tm_q, tm_k, tm_v, tm_la, a, out_f32, stream) != cudaSuccess) {
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_prefill(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                       const float* beta, const float* S0, const int32_t* cu_seqlens, int32_t num_seqs,
                       int64_t total_tokens, int32_t H, int32_t dk, int32_t dv, void* o, float* S_final,
                       void* workspace, size_t workspace_bytes, int32_t* device_status, kda_stream_t stream) {
    return prefill_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv, o,
                        S_final, Snapshots{}, nullptr, workspace, workspace_bytes, device_status, stream);
}

kda_status kda_prefill_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                          const float* beta, const float* S0, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t H, int32_t dk, int32_t dv, void* o, float* S_final,
                          const kda_fusion* fusion, void* workspace, size_t workspace_bytes, int32_t* device_status,
                          kda_stream_t stream) {
    return prefill_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv, o,
                        S_final, Snapshots{}, fusion, workspace, workspace_bytes, device_status, stream);
}

kda_status kda_prefill_snapshots(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                 const float* log_alpha, const float* beta, const float* S0,
                                 const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                 int32_t dk, int32_t dv, void* o, float* S_final, const int32_t* snap_seq,
                                 const int32_t* snap_pos, int32_t num_snaps, float* S_snap, void* workspace,
                                 size_t workspace_bytes, int32_t* device_status, kda_stream_t stream) {
    Snapshots snap;
    snap.seq = snap_seq;
    snap.pos = snap_pos;
    snap.count = num_snaps;
    snap.S = S_snap;
    return prefill_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv, o,
                        S_final, snap, nullptr, workspace, workspace_bytes, device_status, stream);
}


}  // extern "C"

namespace {

// Backward workspace: [schedule][chunk table][forward's bf16 copies and operand images, later the
// backward's per-chunk records][o scratch][snapshot seq][snapshot pos][state after every chunk]
// [adjoint after every chunk].
struct BwdLayout {
    size_t o = 0, seq = 0, pos = 0, snap = 0, xbuf = 0, total = 0;
    int64_t entries = 0;
};
BwdLayout bwd_layout(kda_dtype t, int32_t N, int64_t T, int32_t H) {
    BwdLayout b;
    const WsLayout f = split_layout(t, N, T, H);
    b.entries = max_chunks(N, T);
    const size_t per_state = static_cast<size_t>(b.entries) * H * kHeadDim * kHeadDim * 4;
    const size_t recs = static_cast<size_t>(b.entries) * H * kda::backward_record_bytes();
    b.o = round_up(std::max(f.total, f.copies + recs), kAlign);
    b.seq = b.o + round_up(static_cast<size_t>(T) * H * kHeadDim * esize_of(t), kAlign);
    b.pos = b.seq + round_up(static_cast<size_t>(b.entries) * 4, kAlign);
    b.snap = b.pos + round_up(static_cast<size_t>(b.entries) * 4, kAlign);
    b.xbuf = b.snap + per_state;
    b.total = b.xbuf + per_state;
    return b;
}

// After the plain backward's workspace: the fused prologue's normalised q, k (input dtype), sigmoid beta
// and the inverse norms of q and k, per (token, head).
struct BwdPrologueLayout {
    size_t qh = 0, kh = 0, bh = 0, inv = 0, total = 0;
};
BwdPrologueLayout bwd_prologue_layout(kda_dtype t, int64_t T, int32_t H, size_t plain_total) {
    BwdPrologueLayout p;
    const size_t rows = static_cast<size_t>(T) * H;
    p.qh = round_up(plain_total, kAlign);
    p.kh = p.qh + round_up(rows * kHeadDim * esize_of(t), kAlign);
    p.bh = p.kh + round_up(rows * kHeadDim * esize_of(t), kAlign);
    p.inv = p.bh + round_up(rows * 4, kAlign);
    p.total = p.inv + round_up(rows * 8, kAlign);
    return p;
}

}  // namespace

extern "C" {

size_t kda_prefill_backward_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                            int32_t dk, int32_t dv) {
    if (!ws_args_ok(qkv_dtype, num_seqs, total_tokens, H, dk, dv)) return 0;
    if (!sizes_ok(max_chunks(num_seqs, total_tokens), H, kHeadDim * kHeadDim, 4)) return 0;
    return bwd_layout(qkv_dtype, num_seqs, total_tokens, H).total;
}

size_t kda_prefill_backward_ex_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens,
                                               int32_t H, int32_t dk, int32_t dv) {
    const size_t plain = kda_prefill_backward_workspace_bytes(qkv_dtype, num_seqs, total_tokens, H, dk, dv);
    return plain == 0 ? 0 : bwd_prologue_layout(qkv_dtype, total_tokens, H, plain).total;
}

size_t kda_prefill_backward_gated_workspace_bytes(kda_dtype qkv_dtype, int32_t num_seqs, int64_t total_tokens,
                                                  int32_t H, int32_t dk, int32_t dv) {
    const size_t ex = kda_prefill_backward_ex_workspace_bytes(qkv_dtype, num_seqs, total_tokens, H, dk, dv);
    return ex == 0 ? 0 : round_up(ex, kAlign) + kda::outgate_partial_bytes();
}

}  // extern "C"

namespace {

// The output gate of a gated backward: grad_o is then dL/dy for y = RMSNorm(o) * rms_weight * out_gate.
struct Gate {
    const void* out_gate = nullptr;
    const float* rms_weight = nullptr;  // NULL: ones
    float rms_eps = 0.f;
    float* grad_out_gate = nullptr;
    float* grad_rms_weight = nullptr;  // NULL: not computed
};

// The backward of kda_prefill, optionally through the fused prologue (pre_flags 0 = plain inputs) and the
// output gate (gate NULL = none).
kda_status backward_impl(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                         const float* log_alpha, const float* beta, const float* S0,
                         const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                         int32_t dk, int32_t dv, const void* grad_o, const float* grad_S_final,
                         float* grad_q, float* grad_k, float* grad_v, float* grad_log_alpha,
                         float* grad_beta, float* grad_S0, void* workspace, size_t workspace_bytes,
                         int32_t* device_status, kda_stream_t stream_, uint32_t pre_flags, float l2_eps,
                         const Gate* gate = nullptr) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (qkv_dtype != KDA_DTYPE_BF16 && qkv_dtype != KDA_DTYPE_F32) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || total_tokens > INT32_MAX - 64) return KDA_ERR_INVALID_ARG;
    if (dk != kHeadDim || dv != kHeadDim) return KDA_ERR_UNSUPPORTED;
    const size_t plain_need = kda_prefill_backward_workspace_bytes(qkv_dtype, num_seqs, total_tokens, H, dk, dv);
    if (plain_need == 0 || !sizes_ok(num_seqs, H, kHeadDim, kHeadDim * 4)) return KDA_ERR_INVALID_ARG;
    const BwdPrologueLayout pl = bwd_prologue_layout(qkv_dtype, total_tokens, H, plain_need);
    const size_t gate_part = round_up(pl.total, kAlign);
    const size_t need = gate ? gate_part + kda::outgate_partial_bytes() : pre_flags ? pl.total : plain_need;
    if (!cu_seqlens || !workspace) return KDA_ERR_INVALID_ARG;
    const bool have_tokens = total_tokens > 0;
    if (have_tokens && (!q || !k || !v || !log_alpha || !beta || !grad_o || !grad_q || !grad_k || !grad_v ||
                        !grad_log_alpha || !grad_beta))
        return KDA_ERR_INVALID_ARG;
    if (gate && have_tokens && (!gate->out_gate || !gate->grad_out_gate || !aligned(gate->out_gate, 16) ||
                                !aligned(gate->grad_out_gate, 16)))
        return KDA_ERR_INVALID_ARG;
    if (gate && ((gate->rms_weight && !aligned(gate->rms_weight, 4)) ||
                 (gate->grad_rms_weight && !aligned(gate->grad_rms_weight, 4)) || !(gate->rms_eps >= 0.f)))
        return KDA_ERR_INVALID_ARG;
    if (have_tokens && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, 16) ||
                        !aligned(beta, 4) || !aligned(grad_o, 16) || !aligned(grad_q, 16) || !aligned(grad_k, 16) ||
                        !aligned(grad_v, 16) || !aligned(grad_log_alpha, 16) || !aligned(grad_beta, 4)))
        return KDA_ERR_INVALID_ARG;
    if ((S0 && !aligned(S0, 16)) || (grad_S_final && !aligned(grad_S_final, 16)) ||
        (grad_S0 && !aligned(grad_S0, 16)) || !aligned(workspace, kAlign) || !aligned(cu_seqlens, 4) ||
        (device_status && !aligned(device_status, 4)))
        return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return KDA_ERR_WORKSPACE;

    // Overlap rules: the gradients overlap nothing (each other, the inputs, the workspace).
    const size_t es = esize_of(qkv_dtype);
    const size_t nqk = static_cast<size_t>(total_tokens) * H * kHeadDim;
    const size_t nst = static_cast<size_t>(num_seqs) * H * kHeadDim * kHeadDim;
    const size_t nb = static_cast<size_t>(total_tokens) * H;
    const Range ins[] = {range_of(q, nqk * es),
                         range_of(k, nqk * es),
                         range_of(v, nqk * es),
                         range_of(log_alpha, nqk * 4),
                         range_of(beta, nb * 4),
                         range_of(S0, S0 ? nst * 4 : 0),
                         range_of(cu_seqlens, static_cast<size_t>(num_seqs + 1) * 4),
                         range_of(grad_o, nqk * es),
                         range_of(grad_S_final, grad_S_final ? nst * 4 : 0),
                         range_of(device_status, device_status ? 4 : 0),
                         range_of(gate ? gate->out_gate : nullptr, gate ? nqk * es : 0),
                         range_of(gate ? gate->rms_weight : nullptr, gate && gate->rms_weight ? kHeadDim * 4 : 0)};
    const Range r_ws = range_of(workspace, need);
    const Range outs[] = {range_of(grad_q, have_tokens ? nqk * 4 : 0),
                          range_of(grad_k, have_tokens ? nqk * 4 : 0),
                          range_of(grad_v, have_tokens ? nqk * 4 : 0),
                          range_of(grad_log_alpha, have_tokens ? nqk * 4 : 0),
                          range_of(grad_beta, have_tokens ? nb * 4 : 0),
                          range_of(grad_S0, grad_S0 ? nst * 4 : 0),
                          r_ws,
                          range_of(gate ? gate->grad_out_gate : nullptr, gate && have_tokens ? nqk * 4 : 0),
                          range_of(gate ? gate->grad_rms_weight : nullptr,
                                   gate && gate->grad_rms_weight ? kHeadDim * 4 : 0)};
    constexpr size_t n_outs = sizeof(outs) / sizeof(outs[0]);
    for (size_t i = 0; i < n_outs; ++i) {
        for (const Range& in : ins)
            if (overlap(outs[i], in)) return KDA_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < n_outs; ++j)
            if (overlap(outs[i], outs[j])) return KDA_ERR_INVALID_ARG;
    }

    const kda_status dev = check_device();
    if (dev != KDA_OK) return dev;

    // 0. fused prologue: normalised q, k and sigmoid beta into the workspace's tail
    const int64_t rows = total_tokens * H;
    uint8_t* const wsb = static_cast<uint8_t*>(workspace);
    const bool f32_io = qkv_dtype == KDA_DTYPE_F32;
    const bool norm = (pre_flags & KDA_FUSE_L2NORM_QK) != 0, sig = (pre_flags & KDA_FUSE_BETA_SIGMOID) != 0;
    const void* const qc = norm ? static_cast<const void*>(wsb + pl.qh) : q;
    const void* const kc = norm ? static_cast<const void*>(wsb + pl.kh) : k;
    const float* const bc = sig ? reinterpret_cast<const float*>(wsb + pl.bh) : beta;
    float* const inv = reinterpret_cast<float*>(wsb + pl.inv);
    if (pre_flags && kda::launch_bwd_prologue(f32_io, q, k, beta, wsb + pl.qh, wsb + pl.kh,
                                              reinterpret_cast<float*>(wsb + pl.bh), inv, rows, pre_flags, l2_eps,
                                              stream) != cudaSuccess)
        return KDA_ERR_CUDA;

    // 1. chunk table (validates cu_seqlens into device_status) and a snapshot entry at every chunk end
    const WsLayout fwd = split_layout(qkv_dtype, num_seqs, total_tokens, H);
    const BwdLayout lay = bwd_layout(qkv_dtype, num_seqs, total_tokens, H);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* chunk_off = reinterpret_cast<int32_t*>(ws + fwd.table);
    int32_t* snap_seq = reinterpret_cast<int32_t*>(ws + lay.seq);
    int32_t* snap_pos = reinterpret_cast<int32_t*>(ws + lay.pos);
    float* ckpt = reinterpret_cast<float*>(ws + lay.snap);
    if (kda::launch_chunk_table(cu_seqlens, num_seqs, total_tokens, chunk_off, device_status, nullptr, nullptr, 0,
                                stream) != cudaSuccess ||
        kda::launch_ckpt_entries(cu_seqlens, chunk_off, num_seqs, static_cast<int32_t>(lay.entries), snap_seq,
                                 snap_pos, device_status, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    // 2. the chunkwise prefill records those states (its own table pass rebuilds the same chunk table)
    Snapshots snap;
    snap.seq = snap_seq;
    snap.pos = snap_pos;
    snap.count = static_cast<int32_t>(lay.entries);
    snap.S = ckpt;
    const kda_status fs = prefill_impl(qc, kc, v, qkv_dtype, log_alpha, bc, S0, cu_seqlens, num_seqs, total_tokens,
                                       H, dk, dv, ws + lay.o, nullptr, snap, nullptr, workspace, fwd.total, nullptr,
                                       stream_);
    if (fs != KDA_OK) return fs;
    // 2b. output gate: dL/do over the forward's o, in place (o is dead after this), dL/dgate and dL/dweight
    if (gate && kda::launch_bwd_outgate(f32_io, ws + lay.o, gate->out_gate, grad_o, gate->rms_weight, gate->rms_eps,
                                        ws + lay.o, gate->grad_out_gate, gate->grad_rms_weight,
                                        reinterpret_cast<float*>(ws + gate_part), rows, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    // 3. prep, scan of the adjoint over chunks, value and key kernels
    kda::BackwardArgs a;
    a.q = qc;
    a.k = kc;
    a.v = v;
    a.log_alpha = log_alpha;
    a.beta = bc;
    a.S0 = S0;
    a.cu_seqlens = cu_seqlens;
    a.order = num_seqs > 1 ? reinterpret_cast<const int32_t*>(ws) : nullptr;  // the prefill's schedule
    a.chunk_off = chunk_off;
    a.ckpt = ckpt;
    a.dO = gate ? static_cast<const void*>(ws + lay.o) : grad_o;
    a.dS_final = grad_S_final;
    a.dq = grad_q;
    a.dk = grad_k;
    a.dv = grad_v;
    a.dla = grad_log_alpha;
    a.dbeta = grad_beta;
    a.dS0 = grad_S0;
    a.rec = reinterpret_cast<float*>(ws + fwd.copies);  // the forward's copies and images are dead now
    a.xbuf = reinterpret_cast<float*>(ws + lay.xbuf);
    a.device_status = device_status;
    a.total_tokens = total_tokens;
    a.chunk_slots = lay.entries;
    a.num_seqs = num_seqs;
    a.H = H;
    if (kda::launch_backward(a, f32_io, lay.entries, stream) != cudaSuccess) return KDA_ERR_CUDA;
    // 4. chain rule through the prologue, in place on grad_q, grad_k, grad_beta
    if (pre_flags && kda::launch_bwd_epilogue(f32_io, q, k, reinterpret_cast<const float*>(wsb + pl.bh), inv,
                                              grad_q, grad_k, grad_beta, rows, pre_flags, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_prefill_backward(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                const float* log_alpha, const float* beta, const float* S0,
                                const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                int32_t dk, int32_t dv, const void* grad_o, const float* grad_S_final,
                                float* grad_q, float* grad_k, float* grad_v, float* grad_log_alpha,
                                float* grad_beta, float* grad_S0, void* workspace, size_t workspace_bytes,
                                int32_t* device_status, kda_stream_t stream) {
    return backward_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv,
                         grad_o, grad_S_final, grad_q, grad_k, grad_v, grad_log_alpha, grad_beta, grad_S0, workspace,
                         workspace_bytes, device_status, stream, 0u, 0.f);
}

kda_status kda_prefill_backward_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                   const float* log_alpha, const float* beta, const float* S0,
                                   const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                   int32_t dk, int32_t dv, const void* grad_o, const float* grad_S_final,
                                   float* grad_q, float* grad_k, float* grad_v, float* grad_log_alpha,
                                   float* grad_beta, float* grad_S0, const kda_fusion* fusion, void* workspace,
                                   size_t workspace_bytes, int32_t* device_status, kda_stream_t stream) {
    kda::DecodeFusion fz;
    if (!fusion_ok(fusion, fz, total_tokens > 0)) return KDA_ERR_INVALID_ARG;
    if (fz.flags & KDA_FUSE_OUT_GATE) return KDA_ERR_UNSUPPORTED;
    return backward_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv,
                         grad_o, grad_S_final, grad_q, grad_k, grad_v, grad_log_alpha, grad_beta, grad_S0, workspace,
                         workspace_bytes, device_status, stream, fz.flags, fz.l2_eps);
}

kda_status kda_prefill_backward_gated(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                      const float* log_alpha, const float* beta, const float* S0,
                                      const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                                      int32_t dk, int32_t dv, const void* grad_y, const float* grad_S_final,
                                      float* grad_q, float* grad_k, float* grad_v, float* grad_log_alpha,
                                      float* grad_beta, float* grad_S0, float* grad_out_gate,
                                      float* grad_rms_weight, const kda_fusion* fusion, void* workspace,
                                      size_t workspace_bytes, int32_t* device_status, kda_stream_t stream) {
    kda::DecodeFusion fz;
    if (!fusion || !fusion_ok(fusion, fz, total_tokens > 0) || !(fz.flags & KDA_FUSE_OUT_GATE))
        return KDA_ERR_INVALID_ARG;
    Gate g;
    g.out_gate = fz.out_gate;
    g.rms_weight = fz.rms_weight;
    g.rms_eps = fz.rms_eps;
    g.grad_out_gate = grad_out_gate;
    g.grad_rms_weight = grad_rms_weight;
    return backward_impl(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv,
                         grad_y, grad_S_final, grad_q, grad_k, grad_v, grad_log_alpha, grad_beta, grad_S0, workspace,
                         workspace_bytes, device_status, stream, fz.flags & ~KDA_FUSE_OUT_GATE, fz.l2_eps, &g);
}

}  // extern "C"

namespace {

kda_status decode_impl(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                       const float* beta, float* S, int32_t num_slots, const int32_t* state_indices, int32_t N,
                       int32_t H, int32_t dk, int32_t dv, void* o, const kda_fusion* fusion, int32_t* device_status,
                       kda_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    kda::DecodeFusion fz;
    if (!fusion_ok(fusion, fz, N > 0)) return KDA_ERR_INVALID_ARG;
    if (qkv_dtype != KDA_DTYPE_BF16 && qkv_dtype != KDA_DTYPE_F32) return KDA_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (dk != kHeadDim || dv != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (!sizes_ok(num_slots, H, kHeadDim, kHeadDim * 4) || !sizes_ok(N, H, kHeadDim, 4))
        return KDA_ERR_INVALID_ARG;
    if (static_cast<long long>(N) * H > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return KDA_ERR_INVALID_ARG;
    if (!state_indices && num_slots < N) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, 16) || !aligned(o, 16) ||
        !aligned(S, 16) || !aligned(beta, 4) || (state_indices && !aligned(state_indices, 4)) ||
        (device_status && !aligned(device_status, 4)))
        return KDA_ERR_INVALID_ARG;
    const size_t es = esize_of(qkv_dtype);
    const size_t nio = static_cast<size_t>(N) * H * kHeadDim;
    const Range r_o = range_of(o, nio * es);
    const Range r_s = range_of(S, static_cast<size_t>(num_slots) * H * kHeadDim * kHeadDim * 4);
    const Range inputs[] = {range_of(q, nio * es),
                            range_of(k, nio * es),
                            range_of(v, nio * es),
                            range_of(log_alpha, nio * 4),
                            range_of(beta, static_cast<size_t>(N) * H * 4),
                            range_of(state_indices, state_indices ? static_cast<size_t>(N) * 4 : 0),
                            range_of(device_status, device_status ? 4 : 0)};
    for (const Range& in : inputs)
        if (overlap(r_o, in) || overlap(r_s, in)) return KDA_ERR_INVALID_ARG;
    if (overlap(r_o, r_s)) return KDA_ERR_INVALID_ARG;
    if (fz.flags & KDA_FUSE_OUT_GATE) {
        const Range r_g = range_of(fz.out_gate, nio * es);
        if (overlap(r_g, r_o) || overlap(r_g, r_s)) return KDA_ERR_INVALID_ARG;
    }

    const kda_status dev = check_device();
    if (dev != KDA_OK) return dev;
    if (kda::launch_decode(qkv_dtype == KDA_DTYPE_F32, q, k, v, log_alpha, beta, S, num_slots, state_indices, N, H,
                           o, device_status, stream, fz) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_decode_step(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                           const float* beta, float* S, int32_t num_slots, const int32_t* state_indices, int32_t N,
                           int32_t H, int32_t dk, int32_t dv, void* o, int32_t* device_status,
                           kda_stream_t stream) {
    return decode_impl(q, k, v, qkv_dtype, log_alpha, beta, S, num_slots, state_indices, N, H, dk, dv, o, nullptr,
                       device_status, stream);
}

kda_status kda_decode_step_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                              const float* log_alpha, const float* beta, float* S, int32_t num_slots,
                              const int32_t* state_indices, int32_t N, int32_t H, int32_t dk, int32_t dv, void* o,
                              const kda_fusion* fusion, int32_t* device_status, kda_stream_t stream) {
    return decode_impl(q, k, v, qkv_dtype, log_alpha, beta, S, num_slots, state_indices, N, H, dk, dv, o, fusion,
                       device_status, stream);
}

}  // extern "C"

namespace {

kda_status decode_multi_impl(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                             const float* log_alpha, const float* beta, float* S, int32_t num_slots,
                             const int32_t* state_indices, int32_t N, int32_t T, int32_t H, int32_t dk, int32_t dv,
                             void* o, float* S_steps, const kda_fusion* fusion, int32_t* device_status,
                             kda_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    kda::DecodeFusion fz;
    if (!fusion_ok(fusion, fz, N > 0 && T > 0)) return KDA_ERR_INVALID_ARG;
    if (qkv_dtype != KDA_DTYPE_BF16 && qkv_dtype != KDA_DTYPE_F32) return KDA_ERR_UNSUPPORTED;
    if (N < 0 || T < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (dk != kHeadDim || dv != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (!sizes_ok(num_slots, H, kHeadDim, kHeadDim * 4) || !sizes_ok(N, T, H, kHeadDim * 4) ||
        (S_steps && !sizes_ok(static_cast<int64_t>(N) * T, H, kHeadDim, kHeadDim * 4)))
        return KDA_ERR_INVALID_ARG;
    if (static_cast<long long>(N) * H > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (N == 0 || T == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !S || !o) return KDA_ERR_INVALID_ARG;
    if (!state_indices && num_slots < N) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, 16) || !aligned(o, 16) ||
        !aligned(S, 16) || (S_steps && !aligned(S_steps, 16)) || !aligned(beta, 4) ||
        (state_indices && !aligned(state_indices, 4)) || (device_status && !aligned(device_status, 4)))
        return KDA_ERR_INVALID_ARG;
    const size_t es = esize_of(qkv_dtype);
    const size_t nio = static_cast<size_t>(N) * T * H * kHeadDim;
    const Range r_o = range_of(o, nio * es);
    const Range r_s = range_of(S, static_cast<size_t>(num_slots) * H * kHeadDim * kHeadDim * 4);
    const Range r_st = range_of(S_steps, S_steps ? nio * kHeadDim * 4 : 0);
    const Range inputs[] = {range_of(q, nio * es),
                            range_of(k, nio * es),
                            range_of(v, nio * es),
                            range_of(log_alpha, nio * 4),
                            range_of(beta, static_cast<size_t>(N) * T * H * 4),
                            range_of(state_indices, state_indices ? static_cast<size_t>(N) * 4 : 0),
                            range_of(device_status, device_status ? 4 : 0)};
    for (const Range& in : inputs)
        if (overlap(r_o, in) || overlap(r_s, in) || overlap(r_st, in)) return KDA_ERR_INVALID_ARG;
    if (overlap(r_o, r_s) || overlap(r_o, r_st) || overlap(r_s, r_st)) return KDA_ERR_INVALID_ARG;
    if (fz.flags & KDA_FUSE_OUT_GATE) {
        const Range r_g = range_of(fz.out_gate, nio * es);
        if (overlap(r_g, r_o) || overlap(r_g, r_s) || overlap(r_g, r_st)) return KDA_ERR_INVALID_ARG;
    }

    const kda_status dev = check_device();
    if (dev != KDA_OK) return dev;
    if (kda::launch_decode_multi(qkv_dtype == KDA_DTYPE_F32, q, k, v, log_alpha, beta, S, num_slots, state_indices,
                                 N, T, H, o, S_steps, device_status, stream, fz) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_decode_multi(const void* q, const void* k, const void* v, kda_dtype qkv_dtype, const float* log_alpha,
                            const float* beta, float* S, int32_t num_slots, const int32_t* state_indices, int32_t N,
                            int32_t T, int32_t H, int32_t dk, int32_t dv, void* o, float* S_steps,
                            int32_t* device_status, kda_stream_t stream) {
    return decode_multi_impl(q, k, v, qkv_dtype, log_alpha, beta, S, num_slots, state_indices, N, T, H, dk, dv, o,
                             S_steps, nullptr, device_status, stream);
}

kda_status kda_decode_multi_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                               const float* log_alpha, const float* beta, float* S, int32_t num_slots,
                               const int32_t* state_indices, int32_t N, int32_t T, int32_t H, int32_t dk, int32_t dv,
                               void* o, float* S_steps, const kda_fusion* fusion, int32_t* device_status,
                               kda_stream_t stream) {
    return decode_multi_impl(q, k, v, qkv_dtype, log_alpha, beta, S, num_slots, state_indices, N, T, H, dk, dv, o,
                             S_steps, fusion, device_status, stream);
}

}  // extern "C"
