// attn_internal.h -- declarations shared by the libattn translation units
// (host side only: launch descriptors, tensor-map encoding, error reporting).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "attn.h"

namespace attn {

// Error codes written to the device error word.
enum : int {
    kErrNone = 0,
    kErrTimeoutLoad = 1,     // a consumer waited too long for a TMA tile
    kErrTimeoutSlot = 2,     // the producer waited too long for a free slot
    kErrTimeoutMma = 3,      // a wait on a tensor-core result timed out
    kErrTimeoutSoftmax = 4,  // the MMA issuer waited too long for P
    kErrBadPage = 5,         // a page-table entry in use was outside the page pool
};

// Records a message for attn_last_error() (thread-local) and returns `st`.
attn_status set_error(attn_status st, const char* fmt, ...);

// Launch-configuration trace: with ATTN_TRACE set to anything but "" or "0"
// in the environment, every launch is described on stderr (one line each:
// kernel, grid, block, shared memory, split plan).  Off by default.
bool trace_enabled();
void trace(const char* fmt, ...);

// Device error word (a file-scope __device__ int), as a device pointer.
int* device_error_word();

// Number of SMs of the current device (cached per device).
int sm_count();

// ---- tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point)
// 3-D f16 map over a row-major [S, H, D] tensor: dims (D, H, S), box
// (64, 1, box_rows), 128-byte swizzle (tensor-core operand layout).
attn_status encode_tmap_3d_f16_sw128(CUtensorMap* map, const void* base, int D, int H, int S,
                                     int box_rows);
// Generic map, no swizzle, zero fill.  dims/strides in elements/bytes,
// innermost first; strides[i] is the byte stride of dimension i+1.
attn_status encode_tmap_plain(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes,
                              const uint32_t* box);
// Same, with the 128-byte swizzle (box rows of 128 bytes, as tcgen05 operands read them).
attn_status encode_tmap_sw128(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

// ---- prefill
struct PrefillLaunch {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* lse;
    int S, Hq, Hkv, D, causal, window;
    float softcap, scale;
    int* err_word;
    cudaStream_t stream;
    // chunks over a paged cache (paged != 0): k/v are the page pool
    int paged = 0;
    const int32_t* q_start = nullptr;
    const int32_t* kv_len = nullptr;
    const int32_t* page_table = nullptr;
    int page_size = 0, max_pages = 0, n_pages = 0, B = 0, total_q = 0, max_q = 0;
};
attn_status launch_prefill(const PrefillLaunch& L);

// ---- decode
struct DecodeLaunch {
    const void* q;
    const void* k;
    const void* v;
    const void* k_scales;
    const void* v_scales;
    const int32_t* kv_len;
    const int32_t* page_table;
    int page_size, max_pages, n_pages, max_kv;
    int int8;
    int B, Hq, Hkv, D, window;
    float softcap, scale;
    int split_keys;
    int ring = 0;           // > 0: contiguous ring of `ring` slots, logical token t in slot t % ring
    // tiered decode: 1 = the cold tier (kv_len = cold lengths), 2 = the hot ring
    // (hot token i at index hot_start + i); 0 = a plain decode
    int tier = 0;
    const int32_t* hot_len = nullptr;
    const int32_t* hot_start = nullptr;
    int q_f32 = 0;          // q is f32 [B, Hq, D] (else f16)
    int out_f32 = 0;        // out is f32 [B, Hq, D] (else f16)
    void* out;
    float* lse;
    void* workspace;
    size_t workspace_bytes;
    int* err_word;
    cudaStream_t stream;
};

// Split plan shared by attn_decode_workspace_size and attn_decode.
struct DecodePlan {
    int GH;            // query heads handled together per kv head (1, 2 or 4)
    int HG;            // head groups per kv head: G / GH
    int n_hb;          // head blocks: groups of up to 8 (kv head, head group) units
    int nh_box;        // kv heads covered by one TMA box (the widest head block)
    int split;         // keys per split (multiple of 16)
    long max_items;    // upper bound of work items (sequence, head block, split)
    int n_fix;         // fix-up slots: one per CTA of the balanced kernel (the most it may launch)
    size_t off_tpref, off_fix_meta, off_lse, off_fix_lse, off_o, off_fix_o, bytes;
};
bool make_decode_plan(int B, int Hq, int Hkv, int D, int max_kv, int split_keys, DecodePlan* plan);
attn_status launch_decode(const DecodeLaunch& L, const DecodePlan& plan);
// One-launch decode (decode_direct.cu): a plain decode with the automatic split
// plan whose sequences keep at most 512 keys, with G * D <= 1024 and a small
// cache in all (direct_decode_fits), runs without splits or the combine.
bool direct_decode_fits(const DecodeLaunch& L);
attn_status launch_direct(const DecodeLaunch& L);
attn_status launch_decode_tiered(const DecodeLaunch& cold, const DecodePlan& cold_plan, const DecodeLaunch& hot,
                                 const DecodePlan& hot_plan);

// Test controls of the prefill and decode translation units: the time limit
// of pipeline waits (ns) and the first-tile stall (see ptx.cuh).
attn_status set_test_controls_prefill(unsigned long long wait_limit_ns, int stall);
attn_status set_test_controls_decode(unsigned long long wait_limit_ns, int stall);

constexpr int kDecodeMaxBatch = 4096;
constexpr int kDecodeMaxFix = 256;    // most CTAs the balanced decode kernel launches (>= SMs)

}  // namespace attn
