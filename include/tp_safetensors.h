/*
 * tp_safetensors.h -- shard-on-read straight from a safetensors checkpoint file.
 *
 * "Tensor parallelism" page, §Load a sharded model: from_pretrained() with a
 * tensor-parallel parallel_config has each rank read only its own slice of
 * every weight and place it directly on its device, so no rank ever holds a
 * full-size weight; §Loading performance shows what that saves (load time and
 * peak CPU memory per rank); §Limitations: this loading path reads
 * safetensors weights only.
 *
 * Here one process plays every rank on one GPU (tp.h), so "rank r's slice"
 * is the slice tp_plan_shard() defines, for any range of ranks.  A file is
 * opened once (its header parsed and checked), then each weight is loaded
 * with tp_st_plan_shard_ranks(), which reads the file in one of two ways
 * (tp_st_set_read_mode):
 *   staged: the bytes of the requested ranks' slices are read (pread, several
 *           threads) into a small page-locked staging ring owned by the file
 *           handle, and copied from there into the caller's device shards
 *           while the next part is read;
 *   mapped: where the GPU reads pageable host memory through the host's own
 *           page tables (cudaDevAttrPageableMemoryAccessUsesHostPageTables,
 *           e.g. a Grace host), the file is memory-mapped and the copy engine
 *           reads the slices straight out of the page cache (each range's
 *           pages populated first): no host-side copy, so the load runs at
 *           the CPU-GPU link's rate instead of the host's file-read rate.
 * Staged reads hold two staging buffers of host memory whatever the
 * checkpoint's size.  Mapped reads allocate no host memory for the data, but
 * the pages they read stay mapped into the process until tp_st_close(), so
 * its resident size counts them: they are the page cache's own pages, shared
 * and reclaimable, not copies.  The full weight is never assembled in host or
 * device memory.
 *
 * File format (the published safetensors layout; not defined by the page):
 *   bytes [0, 8)       little-endian uint64 N, the header length;
 *   bytes [8, 8+N)     a UTF-8 JSON object: for each tensor name an object
 *                      {"dtype": "BF16" | ..., "shape": [d0, d1, ...],
 *                       "data_offsets": [begin, end]}, and optionally
 *                      "__metadata__": {string: string};
 *   bytes [8+N, ...)   the data; a tensor's bytes are [begin, end) counted
 *                      from the first byte after the header, row-major, and
 *                      end - begin = product(shape) * element size.
 * tp_st_open() refuses (TP_ERR_FORMAT) a header longer than 100,000,000
 * bytes or running past the end of the file, JSON it cannot parse, an
 * unknown dtype, a missing field, a shape of more than TP_ST_MAX_DIMS
 * dimensions, offsets that are reversed, run past the end of the file or
 * disagree with the shape, tensors whose bytes overlap, and duplicate names.
 * Unknown keys inside a tensor's entry are ignored.
 *
 * Ownership and lifetime: unlike the rest of the library (tp.h), a file
 * handle owns host resources: the open file descriptor, the parsed table and,
 * after the first load, two CUDA events and either two page-locked staging
 * buffers (staged reads) or a read-only mapping of the file plus, for
 * rowwise loads, two device staging buffers of the staging size (mapped
 * reads).  tp_st_close() waits for copies still in flight and releases
 * everything.  A handle is not thread-safe: use one per thread.  Loads are
 * host-synchronous reads feeding asynchronous copies (a mapped load's copies
 * from pageable memory return only when the bytes have left the page cache);
 * they cannot be captured into a CUDA graph.
 */
#ifndef TP_SAFETENSORS_H_
#define TP_SAFETENSORS_H_

#include "tp.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tp_st_file tp_st_file;

#define TP_ST_MAX_DIMS 8
#define TP_ST_DEFAULT_STAGING_BYTES ((size_t)64 << 20) /* per staging buffer; two are used */

typedef enum {
  TP_ST_BOOL = 0,
  TP_ST_U8 = 1,
  TP_ST_I8 = 2,
  TP_ST_F8_E4M3 = 3,
  TP_ST_F8_E5M2 = 4,
  TP_ST_I16 = 5,
  TP_ST_U16 = 6,
  TP_ST_F16 = 7,
  TP_ST_BF16 = 8,
  TP_ST_I32 = 9,
  TP_ST_U32 = 10,
  TP_ST_F32 = 11,
  TP_ST_I64 = 12,
  TP_ST_U64 = 13,
  TP_ST_F64 = 14
} tp_st_dtype;

/* How tp_st_plan_shard_ranks reads the file (see the top of this header). */
typedef enum {
  TP_ST_READ_AUTO = 0,   /* mapped where the current device supports it, else staged (the default) */
  TP_ST_READ_STAGED = 1, /* pread into page-locked staging buffers, then the copy engine */
  TP_ST_READ_MAPPED = 2  /* the copy engine reads a read-only mapping of the file */
} tp_st_read_mode;

/* Bytes per element of a dtype (0 for an unknown value). */
TP_API size_t tp_st_dtype_size(tp_st_dtype dtype);

/*
 * tp_st_open -- open a safetensors file and parse and check its header.
 *
 * path:          file name.
 * staging_bytes: size of each of the two page-locked staging buffers the
 *                loads use (0 = TP_ST_DEFAULT_STAGING_BYTES); rounded up to a
 *                multiple of 4096, at least 4096.  Nothing is allocated until
 *                the first load, so opening and inspecting a file needs no GPU.
 * out:           receives the handle (NULL on failure).
 * Errors: TP_ERR_INVALID_ARG (NULL path or out), TP_ERR_IO (cannot open, stat
 * or read the file), TP_ERR_FORMAT (see above).
 */
TP_API tp_status tp_st_open(const char* path, size_t staging_bytes, tp_st_file** out);

/*
 * tp_st_close -- wait for the handle's copies in flight, free its staging
 * buffers and events, close the file, free the handle.  NULL is a no-op.
 * Returns TP_ERR_CUDA if waiting on a copy reported an error (the handle is
 * released anyway).
 */
TP_API tp_status tp_st_close(tp_st_file* file);

/*
 * tp_st_set_read_mode -- choose how the following loads read the file.
 * Takes effect at the next tp_st_plan_shard_ranks; buffers of the other mode
 * are kept until tp_st_close.  Needs no GPU.
 * Errors: TP_ERR_INVALID_ARG (NULL file, a value outside tp_st_read_mode).
 */
TP_API tp_status tp_st_set_read_mode(tp_st_file* file, tp_st_read_mode mode);

/*
 * tp_st_read_mode_on_device -- the mode a load on the current device would
 * use: TP_ST_READ_STAGED or TP_ST_READ_MAPPED (TP_ST_READ_AUTO resolved).
 * Mapped reads need the device to read pageable memory through the host's
 * page tables and the kernel to populate a mapping on request
 * (MADV_POPULATE_READ, Linux 5.14); the file is mapped by this call if it is
 * not yet.
 * Errors: TP_ERR_INVALID_ARG (NULL argument), TP_ERR_UNSUPPORTED (mode
 * TP_ST_READ_MAPPED where mapped reads are not available), TP_ERR_IO (the
 * mapping failed), TP_ERR_CUDA (no current device).
 */
TP_API tp_status tp_st_read_mode_on_device(tp_st_file* file, tp_st_read_mode* mode);

/* Number of tensors in the file (the "__metadata__" entry is not one); -1 for NULL. */
TP_API int64_t tp_st_count(const tp_st_file* file);

/*
 * tp_st_info -- describe tensor `index` (0 <= index < tp_st_count, in order of
 * increasing data offset).  Any output pointer may be NULL.  *name stays
 * valid until tp_st_close.  shape receives ndim entries (at most
 * TP_ST_MAX_DIMS); offset is the byte offset of the tensor's data from the
 * start of the file; nbytes its length.
 * Errors: TP_ERR_INVALID_ARG for a NULL file or an index out of range.
 */
TP_API tp_status tp_st_info(const tp_st_file* file, int64_t index, const char** name, tp_st_dtype* dtype, int* ndim,
                            int64_t* shape, uint64_t* offset, uint64_t* nbytes);

/* Index of the tensor named `name`, or -1 if there is none (or file/name is NULL). */
TP_API int64_t tp_st_find(const tp_st_file* file, const char* name);

/*
 * tp_st_plan_shard_ranks -- load ranks [rank_begin, rank_begin + rank_count)'s
 * shards of tensor `name` from the file into device buffers.
 *
 * The slice of every rank is tp_plan_shard()'s (tp.h): TP_COLWISE slices
 * dimension 0 and TP_ROWWISE dimension 1, packed blocks (fused_splits) block
 * by block, with the same plan checks in the same order, made before any
 * byte is read.  The tensor is seen as a matrix [rows, cols]: a 2-D tensor as
 * it is; a 1-D tensor (a bias) as [n, 1], so only TP_COLWISE applies to it
 * (a replicated bias is loaded with tp_degree 1); a tensor of three or more
 * dimensions as [d0, d1*d2*...] for TP_COLWISE (TP_ROWWISE on it is
 * TP_ERR_UNSUPPORTED).  Elements are copied as bytes, bit-exact, whatever the
 * dtype.
 *
 * What is read: for TP_COLWISE, exactly the rows of the requested ranks'
 * slices (each rank's part of a block is one contiguous byte range of the
 * file); for TP_ROWWISE, whole rows in chunks of the staging size, from which
 * the requested ranks' columns are extracted on the GPU by the same kernel as
 * tp_plan_shard (the row segments of one rank are short and scattered, so
 * reading whole rows is the faster way even for a single rank).  Mapped
 * reads copy those chunks into a device staging buffer first.
 *
 * dev_outs: host array of rank_count device buffers; dev_outs[i] receives rank
 *           (rank_begin + i)'s dense shard (tp_shard_shape() rows and cols of
 *           the matrix view, times the element size in bytes).
 * stream:   the copies (and, for TP_ROWWISE, the extraction kernel) are
 *           enqueued on it.  The call returns when every byte has been read
 *           from the file and every copy enqueued; the shards are complete
 *           when `stream` reaches that point.
 * Limits: TP_ROWWISE needs one row to fit a staging buffer, and with a 1-byte
 * dtype an even number of columns in every rank's part of every block
 * (TP_ERR_UNSUPPORTED otherwise).
 * Errors: TP_ERR_INVALID_ARG (NULL file/name/dev_outs entry, dev_outs not
 * device memory, a bad rank range), TP_ERR_NOT_FOUND, everything
 * tp_validate() returns, TP_ERR_UNSUPPORTED (also: mode TP_ST_READ_MAPPED
 * where it is not available), TP_ERR_IO (a read failed or came up short; in
 * mapped mode a window that the kernel could not populate), TP_ERR_CUDA.  A
 * plan error leaves device memory untouched; an I/O error part way through
 * leaves the shards partly written.  The file must not be truncated or
 * rewritten while a handle is open on it: mapped loads read its pages in
 * place.
 */
TP_API tp_status tp_st_plan_shard_ranks(tp_st_file* file, const char* name, tp_style style, int tp_degree,
                                        int rank_begin, int rank_count, const int64_t* fused_splits, int n_splits,
                                        int64_t num_heads, int64_t head_dim, void* const* dev_outs,
                                        tp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TP_SAFETENSORS_H_ */
