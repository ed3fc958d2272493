/*
 * wtconv.h -- C ABI of the GB300 WTConv2d library (libwtconv.so).
 *
 * The layer is the wavelet convolution of "Fast and Memory-Efficient Wavelet
 * Convolutions via I/O-Aware Reformulation" (Aflalo, Finder, Amoyal,
 * Treister, Freifeld; arXiv 2608.10805).  Its technical summary on
 * gist.science ("Problem statement", "Methodology") describes it as a
 * drop-in replacement for a depthwise convolution built from: a multi-level
 * 2D Haar analysis; a depthwise k x k convolution of every subband at every
 * level; learned per-channel scales; the L-step synthesis cascade that adds
 * each level's reconstruction to the next finer low-pass band; and a base
 * depthwise convolution with bias, also scaled per channel.  For channel c:
 *
 *   y = s_base[c] * (conv(x, W_base[c]) + b[c]) + sum_l F_l^T Z^l,
 *   Z^l_b = s_w[l,4c+b] * conv(Y^l_b, W_sub[l,4c+b]),   Y^l = F_l x,
 *
 * where F_l is the level-l Haar analysis (orthonormal taps +-1/2; the
 * unconvolved low-pass band feeds the next level; odd sizes are zero-padded
 * on the bottom/right and cropped after synthesis).  Convolutions are
 * stride-1 cross-correlations with zero "same" padding and odd k.  Bands:
 * b = 0 low-pass, 1 row-high (sign (-1)^row), 2 column-high (sign
 * (-1)^column), 3 diagonal; subband channel index 4c+b.
 *
 * The library computes each call on the GPU in one pass over the activations
 * (the pages' "Methodology": the Haar butterflies are recomputed on chip, the
 * multi-level synthesis becomes a single sum whose terms are picked by the
 * bits of each output row and column, the scales are folded into the
 * weights).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates device memory; calls that need scratch take a
 *     caller-provided workspace (size from wtconv_workspace_size).
 *   - Activations x, y, dy, dx are NCHW, contiguous, in desc->dtype.
 *     Parameters and parameter gradients are float32, contiguous:
 *     w_base[C,k,k], b_base[C], w_sub[L,4C,k,k], base_scale[C],
 *     wavelet_scale[L,4C].  Gradients are overwritten, not accumulated.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: no call synchronises the host.
 *   - Arithmetic is float32 (float16/bfloat16 activations are widened on
 *     load and rounded to nearest-even on store).  Results match a float64
 *     evaluation of the unfused layer up to evaluation order.
 *   - Errors: a call validates every argument before it enqueues anything.
 *     On a bad argument it returns an error code and launches nothing.  On a
 *     CUDA launch error it returns WTCONV_ERR_CUDA.  wtconv_last_error()
 *     returns a thread-local message describing the last failure.
 *   - Limits: 3 <= k <= 9, k odd; 1 <= levels <= 8; N >= 0; C, H, W >= 1;
 *     H * W <= 2^24.  Each call keeps whole planes and their pyramids in one
 *     CTA's shared memory when they fit (square planes up to 92..112 px for
 *     wtconv_fwd and wtconv_bwd_data, up to 56 px, or 64 px at levels = 1,
 *     for wtconv_bwd_weight, depending on k and levels).  Larger planes run
 *     in output tiles, each computed from a window of x (or dy) that adds a
 *     halo of 2^levels * (k/2) pixels, rounded up to 8, on every side.  When
 *     that window does not fit one CTA either (levels >= 5 at k >= 5 and
 *     levels >= 6 at k = 3; 16-bit layers at k = 9 from levels = 4), the
 *     layer is computed as two: levels 1..s and the base convolution on the
 *     full planes (s the deepest level count that fits), and levels s+1..L
 *     as a layer of their own, without base convolution, on the float32
 *     level-s low-pass planes (block sums over 2^s x 2^s pixels), whose
 *     output is added back replicated over each block.  The collapsed
 *     synthesis makes this exact up to rounding: for l > s, the coefficient
 *     a pixel takes at level l and its sign bits depend on the pixel only
 *     through (i >> s, j >> s).  Such calls need a workspace in every pass
 *     (wtconv_workspace_size); 16-bit outputs are rounded twice (after the
 *     fine pass and after adding the coarse part).  N = 0 is a valid empty
 *     batch.
 *   - Pointers must be aligned to their element size (WTCONV_ERR_MISALIGNED
 *     otherwise); 16-byte alignment enables vector loads and stores.
 *   - Aliasing: no output (y, dx, a gradient, the workspace) may overlap an
 *     input (x, dy, a parameter) or another output.  Nothing is computed in
 *     place: tiles of large planes read halo pixels that neighbouring tiles
 *     write, and the two passes inside wtconv_bwd's fallback read dy after
 *     dx is written.  The library cannot see buffer lengths and does not
 *     check this; overlapping buffers give undefined results (never an
 *     access outside the buffers).
 */
#ifndef WTCONV_H_
#define WTCONV_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WTCONV_OK = 0,
  WTCONV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, even k, ...           */
  WTCONV_ERR_UNSUPPORTED = 2,  /* valid layer, but outside this build's limits  */
  WTCONV_ERR_MISALIGNED = 3,   /* pointer not aligned to its element size       */
  WTCONV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required    */
  WTCONV_ERR_CUDA = 5          /* a CUDA runtime call or launch failed          */
} wtconv_status_t;

typedef enum { WTCONV_F32 = 0, WTCONV_F16 = 1, WTCONV_BF16 = 2 } wtconv_dtype_t;

typedef enum {
  WTCONV_OP_FWD = 0,
  WTCONV_OP_BWD_DATA = 1,
  WTCONV_OP_BWD_WEIGHT = 2,
  WTCONV_OP_BWD = 3  /* wtconv_bwd: input and parameter gradients in one call */
} wtconv_op_t;

/* Layer geometry.  All fields are plain ints so the layout is fixed. */
typedef struct {
  int N, C, H, W;  /* activation shape, NCHW                                 */
  int levels;      /* L, number of wavelet decomposition levels             */
  int k;           /* kernel size of every depthwise convolution (odd)      */
  int dtype;       /* wtconv_dtype_t of x / y / dy / dx                     */
} wtconv_desc_t;

/* Bytes of device workspace `op` needs for `desc` on the current device (0 if
 * none, or if desc is invalid; the parameter-gradient grid, and with it the
 * size, follows the device's occupancy).  The workspace must be 256-byte
 * aligned; its contents need not be initialised and are garbage after the
 * call.  Packaging: the pages define no such call (their layer is an
 * operator, not an API); it exists because the library never allocates. */
size_t wtconv_workspace_size(const wtconv_desc_t* desc, int op);

/* Forward: y = WTConv2d(x).  b_base may be NULL (no bias).
 * Defined by the technical summary's "Methodology" (fused analysis +
 * depthwise conv, collapsed synthesis, folded scales) and "Problem
 * statement" (drop-in for a depthwise conv).  Needs no workspace (ws may be
 * NULL, ws_bytes 0), except for layers computed as a fine pass plus a coarse
 * layer (see "Limits"): then ws must hold
 * wtconv_workspace_size(desc, WTCONV_OP_FWD) bytes, 256-byte aligned. */
wtconv_status_t wtconv_fwd(const wtconv_desc_t* desc, const void* x, const float* w_base,
                           const float* b_base, const float* w_sub, const float* base_scale,
                           const float* wavelet_scale, void* y, void* ws, size_t ws_bytes,
                           void* stream);

/* Input gradient: dx = A^T dy, where A is the (linear) layer map without the
 * bias.  The summary's "Key contributions" report that the fused
 * implementation reproduces all gradients.  Because the Haar pair is
 * orthonormal and k is odd, A^T is the same fused pass with every kernel
 * rotated by 180 degrees, which is how it is computed.  Workspace as for
 * wtconv_fwd (WTCONV_OP_BWD_DATA). */
wtconv_status_t wtconv_bwd_data(const wtconv_desc_t* desc, const void* dy, const float* w_base,
                                const float* w_sub, const float* base_scale,
                                const float* wavelet_scale, void* dx, void* ws, size_t ws_bytes,
                                void* stream);

/* Parameter gradients for upstream gradient dy at input x:
 *   dw_base[C,k,k], db_base[C] (may be NULL), dw_sub[L,4C,k,k],
 *   dbase_scale[C], dwavelet_scale[L,4C]   (float32, overwritten).
 * The summary's "Key contributions" report that the fused implementation
 * reproduces all parameter gradients; with the scales folded into the
 * weights ("Methodology"), each follows from one correlation sum per weight
 * tap: dW = s * G, ds = <W, G> (+ b * sum dy for the base scale),
 * db = s_base * sum dy, where G correlates the level-l Haar bands of dy with
 * those of x (level 0: the planes themselves).
 * b_base (may be NULL) enters dbase_scale.  Partial correlation sums are
 * reduced in a deterministic order through the workspace, which must hold
 * wtconv_workspace_size(desc, WTCONV_OP_BWD_WEIGHT) bytes. */
wtconv_status_t wtconv_bwd_weight(const wtconv_desc_t* desc, const void* x, const void* dy,
                                  const float* w_base, const float* b_base, const float* w_sub,
                                  const float* base_scale, const float* wavelet_scale,
                                  float* dw_base, float* db_base, float* dw_sub, float* dbase_scale,
                                  float* dwavelet_scale, void* ws, size_t ws_bytes, void* stream);

/* The whole backward in one call: dx (as wtconv_bwd_data) and every parameter
 * gradient (as wtconv_bwd_weight, same arguments and conventions), computed
 * by one kernel that reads x and dy once and builds the Haar pyramid of dy
 * once for both (3 element transfers per element instead of 4).  The
 * summary's "Key contributions" report that the fused implementation
 * reproduces all gradients; merging the two backward passes is this
 * library's.  Results match the two separate calls up to floating-point
 * evaluation order; the parameter gradients are deterministic.  The
 * workspace must hold wtconv_workspace_size(desc, WTCONV_OP_BWD) bytes
 * (256-byte aligned).  Layers the fused kernel does not take run the two
 * separate passes inside this call, with the same results: planes beyond
 * 56 x 56 (depending on k and levels), pyramids whose gradient pass uses
 * 4-row tiles (deep pyramids, small planes packed several per unit; the
 * fused kernel measured no faster there), and layers whose fused working
 * set would leave one CTA per SM.  Errors as for the two calls. */
wtconv_status_t wtconv_bwd(const wtconv_desc_t* desc, const void* x, const void* dy, const float* w_base,
                           const float* b_base, const float* w_sub, const float* base_scale,
                           const float* wavelet_scale, void* dx, float* dw_base, float* db_base, float* dw_sub,
                           float* dbase_scale, float* dwavelet_scale, void* ws, size_t ws_bytes, void* stream);

/* Parameter gradients without a workspace argument, for callers that cannot
 * allocate device memory themselves (for example a plugin inside a host
 * application that owns the whole device-memory budget, or a latency-bound
 * caller that must not call cudaMalloc because it can synchronise the
 * device).  The paper has no counterpart of this call; it is packaging.
 * Same arguments, results and errors as wtconv_bwd_weight, except that the
 * partial sums go to a scratch array of 4 MiB built into the library: a
 * static device array that every GPU which loads the library holds until the
 * process exits.  Layers needing more than 4 MiB of scratch (see
 * wtconv_workspace_size) return WTCONV_ERR_UNSUPPORTED with a message; use
 * wtconv_bwd_weight for them.  Nothing is allocated by this call.
 * Every call outside stream capture looks up the array's device address on
 * the current device (cudaGetSymbolAddress), so the address stays right after
 * a cudaDeviceReset; a call inside a capture uses the address kept from the
 * last call outside one, so make a first call on each device before any
 * capture (and again after a reset), else the call returns
 * WTCONV_ERR_INVALID_ARG.  All calls share the one array and it keeps the last
 * call's contents (every entry is rewritten before use, so nothing needs
 * clearing): calls that can overlap on the GPU -- on different streams, or
 * from different host threads -- race on it and must be serialised by the
 * caller. */
wtconv_status_t wtconv_bwd_weight_noalloc(const wtconv_desc_t* desc, const void* x, const void* dy,
                                          const float* w_base, const float* b_base, const float* w_sub,
                                          const float* base_scale, const float* wavelet_scale,
                                          float* dw_base, float* db_base, float* dw_sub,
                                          float* dbase_scale, float* dwavelet_scale, void* stream);

/* Static name of a status code.  Packaging (no counterpart in the pages). */
const char* wtconv_status_string(wtconv_status_t status);

/* Thread-local description of the last failure on this thread ("" if none).
 * Packaging (no counterpart in the pages). */
const char* wtconv_last_error(void);

/* Packaging (no counterpart in the pages): the number of in-kernel waits on
 * the current device that gave up since the previous call, then resets the
 * count.  The kernels wait for their own
 * asynchronous (TMA and bulk) plane copies with a time limit of about a second; a
 * wait that runs out records itself here and the kernel stops early (its
 * outputs are then invalid).  0 in normal operation.  Synchronises the
 * current device. */
unsigned int wtconv_device_faults(void);

/* Test support, off by default (no counterpart in the pages): with enable
 * nonzero, every later call on any thread gives the in-kernel waits for its
 * plane copies a limit of about 2^20 clock cycles and arms each copy's
 * barrier with 16 bytes more than the copy delivers, so each such wait runs
 * out: the kernel records the fault (see wtconv_device_faults), lets its copy
 * land and leaves early, with its outputs invalid and the device usable.
 * This exercises the give-up path of the bounded waits without a GPU fault.
 * enable = 0 restores normal operation. */
void wtconv_test_copy_timeout(int enable);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_H_ */
