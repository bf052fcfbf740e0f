/*
 * cp.h -- C ABI of libcp, the GB300 (sm_103a) lookup-decode for Conditional
 * Program (CP) compressed memory tables.
 *
 * Method (pages cited by title):
 *   [P4] "2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다"
 *        (onedev.kr/papers/1189)
 *   [P1] "Two-bit lookup tables shrink DeepSeek's 203 GB memory to 51 GB and
 *        cut prefill from 64.66 s to 13.27 s" (ai4snews.wisdomeyes.cn)
 *
 * Each table row i is one independently addressable record holding a b-bit-per-
 * coordinate code c_i and a 16-bit scale alpha_i, b + 16/d bits per parameter;
 * the reconstruction rule f is shared by the whole table and applied only to
 * rows that are looked up: e_hat_i = alpha_i * f(c_i) [P4 section 어떻게 동작하나
 * "how it works"].  The runtime fetches only the requested records, restores
 * them with a fused kernel and hands them over in the original lookup order
 * [P4 section 무엇과 다른가 "how it differs"].  The table can sit in GPU HBM or
 * in pinned host DRAM read over the host link [P4 section 전제와 한계
 * "assumptions and limits"; P1 "Interpretation"].
 *
 * Format constants (the pages leave them open; fixed here once):
 *   V = 2 coordinates per trellis step; k = 2b bits per step, k in {3,4,5,6}
 *   (b = 1.5, 2, 2.5, 3); T = d/2 steps; Lc = k*T code bits per row.
 *   Code bit j = (code[j >> 3] >> (j & 7)) & 1 (LSB first, little-endian bytes).
 *   State s_t = the 16 code bits ending at bit k(t+1), oldest bit lowest, bit
 *   positions taken mod Lc (tail-biting).
 *   h = s*s + s (mod 2^32); (y0, y1) = LUT[(h >> 14) & 511]; y1 = -y1 when bit
 *   23 of h is set.  LUT: 512 fp16 pairs, shared by the table.
 *   out[2t] = bf16_rn(float(alpha) * y0), out[2t+1] = bf16_rn(float(alpha) * y1):
 *   one fp32 product (exact), one round-to-nearest-even to bf16.
 *
 * Record (AoS) layout, R = d*k/16 + 2 bytes, no padding:
 *   [ code: d*k/16 bytes ][ alpha: bf16, little-endian ]
 * Record i starts at byte i*R of the records buffer (2-byte aligned in general).
 *
 * Conventions for every call:
 *   - Stream-ordered and asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  The decode calls (cp_lookup_decode,
 *     cp_lookup_decode_host, cp_lookup_decode_reduce) queue kernels only: they
 *     never synchronise or allocate, so they can be captured into a CUDA graph
 *     and replayed (with new ids written into the captured buffers).  The calls
 *     that synchronise `stream` say so: cp_get_status, cp_table_load_mixed,
 *     cp_table_set_cache and cp_encode_rows.
 *   - Argument errors are detected on the host and returned before any work is
 *     queued; nothing is written in that case.
 *   - The caller owns every large buffer (records, SoA copy, ids, output); a
 *     table handle borrows them and they must outlive it.  The handle owns only
 *     its LUT copy, its device status word, its geometry and, for host-resident
 *     tables, 8.4 MB of device scratch for the visiting order.
 *   - Out-of-range ids never fault: the output row is written as zeros and the
 *     table's device status word records CP_ERR_INDEX_OOB for cp_get_status.
 *   - n = 0 is a valid no-op.
 *   - Geometry accepted by the CUDA path: d % 8 == 0, 8 <= d <= 4096,
 *     (d*k) % 32 == 0 (a record is a whole number of 16-bit words, so every
 *     record starts 2-byte aligned), 1 <= n_rows <= 2^40.
 */
#ifndef CP_H_
#define CP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cp_table cp_table; /* opaque handle */

typedef enum cp_status {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1, /* bad pointer, alignment, geometry or residency */
  CP_ERR_INDEX_OOB = 2,   /* a previous decode saw an id outside [0, n_rows) */
  CP_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  CP_ERR_NO_MEMORY = 4,   /* the handle's own small allocations failed */
  CP_ERR_FORMAT = 5       /* LUT or record contents unusable (non-finite LUT) */
} cp_status;

enum { CP_LAYOUT_AOS = 0, CP_LAYOUT_SOA = 1 };
enum { CP_RESIDENT_DEVICE = 0, CP_RESIDENT_HOST = 1 };

/* Bytes of one AoS record: d*k/16 code bytes + 2 (the bf16 scale); this is
 * exactly b + 16/d bits per parameter [P4 "how it works"].  0 if the geometry
 * is not accepted. */
uint64_t cp_record_bytes(uint32_t d, uint32_t bits_per_step);

/* Bytes a caller must provide for the SoA copy of an n_rows table:
 * codes[n_rows][S] with S = d*k/16 rounded up to 16, then alpha[n_rows] (bf16),
 * the alpha array starting at byte n_rows*S and padded to a multiple of 16.
 * 0 if the geometry is not accepted. */
uint64_t cp_soa_bytes(uint64_t n_rows, uint32_t d, uint32_t bits_per_step);

/*
 * cp_table_load -- bind a compressed table (records in the AoS layout above)
 * to a handle, validate its geometry, copy the shared LUT to the device and,
 * for CP_LAYOUT_SOA, repack the records on the device into `soa_dst`.
 *
 *   out           receives the handle (set to NULL on error).
 *   records       AoS records, n_rows * R bytes, 16-byte aligned.  The buffer
 *                 must span all n_rows * R bytes: the kernels read up to its
 *                 last byte and this call cannot check the size of a pointer.
 *                 CP_RESIDENT_DEVICE: device memory.
 *                 CP_RESIDENT_HOST: host memory, page-locked by the caller
 *                 (cudaHostAlloc, or cudaHostRegister).  If it is plain pageable
 *                 memory, the call registers it (mapped, read-only) and the
 *                 handle unregisters it in cp_table_free.
 *   n_rows, d, bits_per_step: the geometry (k = 2b).
 *   lut_fp16      host pointer to 512 x (y0, y1) fp16 bit patterns (2048 bytes),
 *                 copied during the call; every entry must be finite.
 *   residency     CP_RESIDENT_DEVICE or CP_RESIDENT_HOST.
 *   layout        CP_LAYOUT_AOS: the decoder reads `records` in place.
 *                 CP_LAYOUT_SOA: the decoder reads `soa_dst` (cp_soa_bytes
 *                 bytes, 16-byte aligned, device memory, or for a host-resident
 *                 table pinned host memory) which this call fills, stream-ordered.
 *   soa_dst       NULL for CP_LAYOUT_AOS.
 *   stream        cudaStream_t for the LUT copy and the repack.
 * The handle is usable by later work on `stream` (or on any stream after it has
 * been synchronised).
 */
cp_status cp_table_load(cp_table** out, const void* records, uint64_t n_rows, uint32_t d,
                        uint32_t bits_per_step, const uint16_t* lut_fp16, int residency,
                        int layout, void* soa_dst, void* stream);

/*
 * cp_table_load_mixed -- bind a table whose rows have different code rates
 * (frequency-based bit allocation, tried on [P4 "assumptions and limits"]):
 * record r, [code at k_r bits per step][bf16 alpha], occupies bytes
 * [offsets[r], offsets[r+1]) of `records`, and k_r = (R_r - 2) * 16 / d must be
 * 3, 4, 5 or 6.  Device-resident, AoS.
 *   records  device, offsets[n_rows] bytes, 16-byte aligned.
 *   offsets  device uint64[n_rows + 1], offsets[0] = 0, even, increasing;
 *            borrowed for the handle's lifetime.
 *   d        multiple of 32 in [32, 4096].
 * The call checks every record length on the device and synchronises `stream`;
 * CP_ERR_FORMAT if one gives no valid rate.  cp_lookup_decode then decodes the
 * table (per-row rate); cp_lookup_decode_reduce and the SoA layout do not apply.
 */
cp_status cp_table_load_mixed(cp_table** out, const void* records, const uint64_t* offsets,
                              uint64_t n_rows, uint32_t d, const uint16_t* lut_fp16, void* stream);

/*
 * cp_lookup_decode -- e_hat_j = alpha_{r_j} * f(c_{r_j}) for the n requested
 * row ids r_j = idx[j], written as bf16 rows in lookup order, duplicates
 * included [P4 "how it differs"].  The table must be CP_RESIDENT_DEVICE.
 *
 *   idx   device pointer, n int64 row ids, 8-byte aligned.
 *   out   device pointer, bf16 [n][d] row-major (n*d*2 bytes), 16-byte aligned.
 *         It may also be page-locked host memory that the device can address
 *         (cudaHostAlloc, or cudaHostRegister with mapping; with unified
 *         addressing the host pointer is the device pointer): the kernel then
 *         writes the rows over the host link, with no separate copy.
 * Out-of-range ids give zero rows and set the status word (see cp_get_status).
 * Launch (single-rate table): one kernel of ceil(n / 32) CTAs of 256 threads
 * (32 lookups per CTA), each with 4 KB (d = 256, 512) or 8 KB of LUT plus 32
 * record stages of shared memory (under 18 KB at d = 1024, b = 2); work from
 * other streams can share the SMs.  A mixed-rate table runs the same grid shape (with stages sized for
 * the widest rate) and resolves each id to its record's offset and rate inside
 * the kernel.
 */
cp_status cp_lookup_decode(const cp_table* t, const int64_t* idx, uint64_t n, uint16_t* out,
                           void* stream);

/*
 * cp_lookup_decode_host -- the same operation for a CP_RESIDENT_HOST table: the
 * kernel reads only the requested records directly from pinned host DRAM over
 * the host link (zero-copy) [P4 "assumptions and limits"; P1 "Interpretation"].
 * idx and out are device pointers as for cp_lookup_decode; the output is the
 * same, bit for bit, as cp_lookup_decode on the same records.
 * Internally, per pass of at most 2^20 lookups, the lookups are visited
 * grouped by row-id range (a counting partition into 4096 ranges), so that
 * successive host reads are close in the host address space; every row is still
 * written at its own position.  Each SM takes one contiguous slice of that
 * order; the repeats of an id fall into the same slice and find the record in
 * that SM's L1 cache (on a 196,608-lookup Zipf replay, about 1.03 fetches per
 * distinct id cross the host link, against 2.2 for one fetch per lookup).
 * This state lives in 8.4 MB of device scratch owned by
 * the handle (allocated by cp_table_load), so calls on one host-resident handle
 * must be ordered on one stream (or otherwise serialised).
 */
cp_status cp_lookup_decode_host(const cp_table* t, const int64_t* idx, uint64_t n,
                                uint16_t* out, void* stream);

/*
 * cp_table_set_cache -- frequency-based caching for a host-resident table: keep
 * device copies of the records of `m` hot rows, so that cp_lookup_decode_host
 * reads them from HBM instead of over the host link.  The pages name access
 * counts as the input of frequency-based caching [P1 "Perspective"; P4
 * "assumptions and limits"]; the caller chooses the rows (e.g. the most
 * frequent ids of past traffic).
 *   hot_rows  host pointer, m distinct ids in [0, n_rows) (any order).
 *   cache     device buffer of m * R bytes, 16-byte aligned, owned by the caller;
 *             it receives the records (AoS, ascending row order).
 *   m = 0     removes the cache.  Replacing a cache synchronises `stream` first.
 * The call allocates the cache map (2^ceil(log2(2m)) slots of 12 bytes plus
 * 8m bytes, owned by the handle) and returns after the cache is built (it
 * synchronises `stream`).  Output of cp_lookup_decode_host is unchanged, bit for
 * bit.  Host-resident AoS tables with d = 256, 512 or 1024; otherwise
 * CP_ERR_INVALID_ARG.  Not to be called while decodes on the handle are in
 * flight on other streams.
 */
cp_status cp_table_set_cache(cp_table* t, const int64_t* hot_rows, uint64_t m, void* cache,
                             void* stream);

/*
 * cp_lookup_decode_reduce -- lookup-decode fused with a weighted readout.  The
 * pages hand the restored rows to "the existing readout" [P4 "how it differs"];
 * this synthetic readout sums each group of `group` consecutive lookups (for
 * example the rows one token gathers in one layer), so only one row per group
 * leaves the kernel:
 *   out[g][q] = bf16_rn(acc),  acc = fmaf(w[g*group + i], float(row_i[q]), acc)
 * for i = 0 .. group-1 in order, acc starting at +0 (fp32), where row_i is the
 * bf16 row cp_lookup_decode would write for idx[g*group + i] (zeros for an
 * out-of-range id, which also sets the status word) and w = 1 when weights is
 * NULL.
 *   idx      device, n_groups * group int64 ids.
 *   weights  device fp32 [n_groups * group], or NULL.
 *   out      device bf16 [n_groups][d], 16-byte aligned.
 * Device-resident tables with d in {256, 512, 1024}; otherwise CP_ERR_INVALID_ARG.
 */
cp_status cp_lookup_decode_reduce(const cp_table* t, const int64_t* idx, uint64_t n_groups,
                                  uint32_t group, const float* weights, uint16_t* out,
                                  void* stream);

/*
 * cp_encode_rows -- offline compression on the GPU: rows e -> AoS records.
 * z = sqrt(d) e / |e| is coded by the tail-biting trellis (TCQ) and
 * alpha = |e|_2 / |f(c)|_2 restores the norm [P4 "how it differs"].  Search:
 * a free-start Viterbi on the sequence rotated by T/2 steps picks the 16 - k
 * pre-window bits from its best path, then one Viterbi constrained to them
 * gives a valid tail-biting code (the exact search, over every pre-window, is
 * 2^(16-k) times costlier).  Precision (the pages fix none): |e|, z and alpha in
 * fp64 with sums in index order, path metrics in fp32 (branch cost
 * fl(fl((z0-y0)^2) + fl((z1-y1)^2)), no fused multiply-add); survivor per group
 * of states sharing predecessors: smallest metric, then smallest dropped bits;
 * final state: smallest metric, then smallest state.  A zero row gives a zero
 * record.  Rows must be finite.
 *   e        device fp32 [rows][d].
 *   lut_fp16 host, 512 x (y0, y1) fp16 patterns (finite).
 *   records  device, rows * R bytes (R = d*k/16 + 2).
 *   cost     device fp32 [rows] (optional): the search's path metric.
 * Runs one 4-CTA thread-block cluster per row in flight.  Allocates and frees
 * its workspace (d/2 * 2^(16-k) traceback bytes per cluster in flight, 2 MB at
 * d = 1024, k = 4) and synchronises `stream` before returning.  d >= 16.
 * Errors: CP_ERR_INVALID_ARG (pointers, geometry), CP_ERR_FORMAT (LUT),
 * CP_ERR_NO_MEMORY (workspace), CP_ERR_CUDA (launch or cluster occupancy).
 */
cp_status cp_encode_rows(const float* e, uint64_t rows, uint32_t d, uint32_t bits_per_step,
                         const uint16_t* lut_fp16, uint8_t* records, float* cost, void* stream);

/*
 * cp_encode_workspace_bytes -- device workspace that cp_encode_rows_ws needs for
 * `rows` rows of this geometry on the current device (traceback bytes of every
 * cluster in flight plus 2 KB for the LUT); 0 for a rejected geometry or when
 * the device cannot run the encoder's clusters.
 */
uint64_t cp_encode_workspace_bytes(uint64_t rows, uint32_t d, uint32_t bits_per_step);

/*
 * cp_encode_rows_ws -- cp_encode_rows with a caller-owned workspace: it queues
 * the LUT copy and the encoder kernel on `stream` and returns without
 * synchronising or allocating, so the kernel can be timed with events and
 * repeated calls reuse one workspace.  Same arguments and results as
 * cp_encode_rows, plus
 *   workspace        device memory, 256-byte aligned, at least
 *                    cp_encode_workspace_bytes(rows, d, bits_per_step) bytes;
 *                    used until the queued work completes (calls sharing it
 *                    must be ordered on one stream).
 *   workspace_bytes  its size; CP_ERR_INVALID_ARG when too small.
 */
cp_status cp_encode_rows_ws(const float* e, uint64_t rows, uint32_t d, uint32_t bits_per_step,
                            const uint16_t* lut_fp16, uint8_t* records, float* cost,
                            void* workspace, uint64_t workspace_bytes, void* stream);

/*
 * cp_get_status -- synchronise `stream`, then report and clear the table's
 * device status word: CP_ERR_INDEX_OOB if any decode since the last call saw an
 * out-of-range id, CP_ERR_CUDA if the stream holds a CUDA error, else CP_OK.
 */
cp_status cp_get_status(const cp_table* t, void* stream);

/*
 * cp_lookup_decode_host_noalloc -- cp_lookup_decode_host for callers that
 * cannot allocate device memory.  (The pages have no counterpart: this is an
 * integration entry point of this library.)
 *
 * Who needs it: code whose device memory belongs to one pool allocator (a
 * plugin may not call cudaMalloc behind the owner's back), code that must not
 * call cudaMalloc/cudaFree while other streams run (both can synchronise the
 * device), or a runtime that fixes its memory budget up front.  cp_table_load
 * allocates, so such callers pass everything themselves:
 *   records   pinned, mapped host memory holding n_rows AoS records (16-byte
 *             aligned; page-locked by the caller, e.g. cudaHostAlloc).  It must
 *             span n_rows * R bytes: the kernels may read up to its last byte
 *             over the host link, and the library cannot check the size.
 *   n_rows, d, bits_per_step: geometry as for cp_table_load.
 *   lut_fp16  host pointer, 512 x (y0, y1) fp16 patterns, finite.
 *   idx       device, n int64 ids;  out: device bf16 [n][d], 16-byte aligned.
 *   status    device uint32 owned by the caller: bit 0 is OR-ed in when an id is
 *             out of range (clear it yourself before the call if needed).
 * It allocates nothing: its scratch (the LUT copy, the range counts, the visiting
 * order) is one static device array of about 0.56 MB that every GPU loading the
 * library holds until the process exits.  Limit: n <= 65536 lookups per call;
 * larger n returns CP_ERR_INVALID_ARG before any work is queued.
 * The first call on a device looks up that array's device address and clears
 * its counters with a synchronous memset (once per device, so that first call
 * synchronises the device).  The address is kept for the life of the process: after cudaDeviceReset it no longer names the
 * array, so do not call this entry point on a device that has been reset.  All calls share the
 * array and it keeps the last call's contents (each call clears what must start
 * empty), so calls that overlap on the GPU (on different streams, or from
 * different threads without ordering) race: order them on one stream.
 * The output equals cp_lookup_decode_host's bit for bit.
 */
cp_status cp_lookup_decode_host_noalloc(const void* records, uint64_t n_rows, uint32_t d,
                                        uint32_t bits_per_step, const uint16_t* lut_fp16,
                                        const int64_t* idx, uint64_t n, uint16_t* out,
                                        uint32_t* status, void* stream);

/*
 * cp_measure_stream_read -- read `bytes` bytes of `buf` once with a streaming
 * kernel (16-byte loads, grid-stride, four loads in flight per thread; nothing
 * observable is written).  Timed with events on `stream`, it gives the
 * bandwidth that bounds a lookup-decode: read zero-copy from page-locked host
 * memory it is the host link's rate (the roofline of cp_lookup_decode_host,
 * beside a cudaMemcpyAsync from the same memory); from device memory it is the
 * HBM read rate.  The pages give the host link only as the path of the slow
 * placement [P4 "assumptions and limits"]; this measures it on the machine.
 *   buf    device memory, or page-locked host memory the device can address;
 *          16-byte aligned.
 *   bytes  a positive multiple of 16.
 * CP_ERR_INVALID_ARG for any other buffer; queues one kernel, no allocation.
 */
cp_status cp_measure_stream_read(const void* buf, uint64_t bytes, void* stream);

/*
 * cp_measure_record_read -- read the records rows[0..n) of a record table once,
 * each as the 16-byte pieces that cover it (the host path's own loads), with no
 * decode and nothing observable written.  Timed with events on `stream` with
 * the distinct ids of a replay, sorted, it gives the rate at which the host link
 * delivers whole records at scattered addresses: the roofline of
 * cp_lookup_decode_host's access pattern, below the streaming rate because a
 * 258-byte record at a 2-byte boundary spans nine 32-byte sectors.  The pages
 * place the table in pinned host DRAM as the slow placement [P4 "assumptions
 * and limits"]; this measures that placement's record rate on the machine.
 *   table         device memory or mapped page-locked host memory, 16-byte
 *                 aligned, table_bytes long (at least one record).
 *   record_bytes  bytes per record (R); record r starts at byte r * R.
 *   rows, n       device array of n int64 row ids (0 < n < 2^48), 8-byte
 *                 aligned; ids at or past table_bytes / R are skipped.
 * CP_ERR_INVALID_ARG for any other argument; queues one kernel, no allocation.
 */
cp_status cp_measure_record_read(const void* table, uint64_t table_bytes, uint32_t record_bytes,
                                 const int64_t* rows, uint64_t n, void* stream);

/* Release what the handle owns (LUT copy, status word, host registration made
 * by cp_table_load).  Borrowed buffers are untouched.  NULL is a no-op. */
void cp_table_free(cp_table* t);

/* Static string for a status code. */
const char* cp_status_string(cp_status s);

/* Text of the last CUDA error seen by this library on the calling thread ("" if
 * none). */
const char* cp_last_error(void);

/* Test hook for failure handling on the host: the next `count` calls of the
 * chosen kind fail as if the CUDA runtime had refused them
 * (1 = device allocation, 2 = host registration / device alias).  Returns
 * CP_ERR_INVALID_ARG for an unknown kind. */
cp_status cp_test_inject_failure(int kind, int count);

#ifdef __cplusplus
}
#endif

#endif /* CP_H_ */
