/*
 * gs.h -- C ABI of the GB300 3D Gaussian Splatting training-step library (libgs.so).
 *
 * One training step over a batch of B views is, per view:
 *   gs_project -> gs_bin_sort -> gs_render_fwd -> gs_loss -> gs_render_bwd -> gs_project_bwd
 * and, once per batch, gs_visible_sets -> gs_sparse_adam (or, fusing the per-view
 * gs_project_bwd calls with the update, gs_project_bwd_adam once per batch).
 * The step follows the training flow of the Grendel-GS notes ("训练流程": transform,
 * render by depth-sorted alpha compositing, L1 + SSIM loss, backpropagation, update)
 * with the visible-only update of the Odin summary ("研究背景与动机": a view renders,
 * backpropagates and updates only the primitives it sees).
 *
 * Conventions shared by every entry point
 *  - All array arguments are DEVICE pointers owned by the caller unless a comment says
 *    "host".  The library never allocates device memory in these calls: scratch comes
 *    from a caller workspace sized by the matching *_workspace_size() call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) unless it says it synchronises.
 *  - Arrays of float4 records must be 16-byte aligned; 64-bit arrays 8-byte aligned.
 *  - Returns GS_OK, or an error code with a message readable by gs_last_error() (per
 *    host thread).  Argument errors are detected on the host before anything is enqueued.
 *  - Layouts (float32, plane-major):
 *      params  [15][N][4]  p0 = (x, y, z, opacity logit), p1 = (log s0, log s1, log s2, 0),
 *                          p2 = quaternion (w, x, y, z), p3..p14 = SH sh[k][c] flattened as
 *                          3k + c (k = 0..15 degree<=3 coefficients, c = r, g, b), four per
 *                          plane -- the 59-float record of the Grendel-GS parameter table.
 *      proj    [3][N][4]   q0 = (u, v, depth z, opacity), q1 = (conic A, B, C, radius as int32
 *                          bits), q2 = (r, g, b, tiles touched as int32 bits).  A culled
 *                          Gaussian has radius 0 and tiles 0.
 *      grad2d  [N][12]     (du, dv, dopacity, 0, dA, dB, dC, 0, dr, dg, db, 0).
 *      image   [3][H][W]   channel-major; T_final and n_contrib are [H][W].
 *  - Pixel (px, py) is sampled at (px + 0.5, py + 0.5); tiles are 16 x 16 pixels
 *    (Grendel-GS notes §1.2), numbered row-major, Tx = ceil(W/16), Ty = ceil(H/16).
 */
#ifndef GS_H_
#define GS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GS_OK = 0,
  GS_ERR_INVALID = 1,   /* null pointer, misalignment, negative size, bad dimensions */
  GS_ERR_CUDA = 2,      /* a CUDA runtime call failed; message from cudaGetErrorString */
  GS_ERR_CAPACITY = 3,  /* the instance count exceeds the caller's capacity */
  GS_ERR_TIMEOUT = 4    /* a bounded device-side wait gave up (see gs_bin_sort) */
} gs_status;

/* Pinhole camera, OpenCV axes (x right, y down, z forward).  p_cam = R p_world + t,
 * R row-major.  u = fx x/z + cx, v = fy y/z + cy.  Gaussians with z <= znear are culled. */
typedef struct {
  float R[9];
  float t[3];
  float fx, fy, cx, cy, znear;
  int32_t width, height;
} gs_camera;

/* Message of the last failing call on this host thread ("" if none). */
const char* gs_last_error(void);

/* Library ABI version (increments when a signature changes). */
int gs_version(void);

/* ---------------------------------------------------------------------------
 * gs_project -- per-Gaussian projection ("transform" step: 3D Gaussian -> screen
 * position, depth, footprint radius, colour; Grendel-GS notes, 训练流程).
 * For Gaussian i of params [15][n][4], writes proj [3][n][4]:
 *   cull if z <= znear; s = exp(log s); opacity = sigmoid(logit); q normalised;
 *   Sigma = R(q) diag(s^2) R(q)^T; J = perspective Jacobian at the camera-space point
 *   with x/z, y/z clamped to +-1.3 tan(fov/2); Sigma2D = J R Sigma R^T J^T + 0.3 I;
 *   conic = Sigma2D^-1 (cull if det <= 0); radius = ceil(3 sqrt(lambda_max));
 *   tile rectangle [floor((u-r)/16), floor((u+r)/16)+1) clamped to the grid (cull if
 *   empty); colour = max(0, sum_k sh[k] Y_k(dir) + 0.5) with dir the unit vector from
 *   the camera centre to the mean and Y_k the real degree-3 SH basis.
 * n == 0 is a no-op.
 */
gs_status gs_project(const float* params, int64_t n, const gs_camera* cam, float* proj, void* stream);

/* gs_project_batch -- gs_project for the `batch` views of one training step (the Grendel-GS
 * notes' batch of images, §4.2), results identical to `batch` gs_project calls.  One launch
 * per 16 views reads each Gaussian's parameters once and computes the view-independent part
 * (scales, opacity, rotation, 3-D covariance) once.
 *   cams   host array of `batch` cameras.
 *   projs  host array of `batch` device pointers, [3][n][4] each, 16-byte aligned.
 *   visible_bits  optional (NULL: not written), [batch][bits_stride] uint32: bit i % 32 of
 *          word i / 32 of view b set iff Gaussian i has radius > 0 in view b (bits past n
 *          clear); bits_stride >= ceil(n / 32).  The visible sets' input (gs_visible_sets).
 * batch must be >= 1; n == 0 is a no-op.
 */
gs_status gs_project_batch(const float* params, int64_t n, const gs_camera* cams, int batch,
                           float* const* projs, uint32_t* visible_bits, int64_t bits_stride, void* stream);

/* ---------------------------------------------------------------------------
 * gs_bin_sort -- tile binning and depth sort ("find the Gaussians covering a pixel,
 * sort by depth"; Grendel-GS notes, 训练流程, with 16x16 tiles, §1.2).
 * Every Gaussian with radius > 0 is duplicated once per tile of its rectangle
 * (Gaussian index ascending, tiles row-major within the rectangle) with
 *   key = (tile id << 32) | float bits of z,  value = Gaussian index,
 * and the M instances are stably radix-sorted by key, i.e. ordered by (tile, depth,
 * index).  ranges[2t], ranges[2t+1] = [start, end) of tile t in the sorted arrays,
 * [0, 0) for an empty tile.
 *   proj       [3][n][4] from gs_project.
 *   workspace  gs_bin_sort_workspace_size(n, capacity, cam) bytes, 256-byte aligned.
 *   keys, vals outputs of `capacity` entries; keys may be NULL (not written: the
 *              tile ranges and the values are all that compositing reads).
 *   ranges     output, 2 * Tx * Ty uint32.
 *   count      device int64[2]: count[0] = M (the true count even when it exceeds
 *              capacity), count[1] = status bits (0 = ok, 1 = capacity exceeded,
 *              2 = a bounded device-side wait gave up).  On any nonzero status the outputs are
 *              not valid and ranges are left empty.
 *   count_host optional host int64: if non-NULL the call synchronises the stream, stores
 *              M there, and returns GS_ERR_CAPACITY / GS_ERR_TIMEOUT per count[1].
 * capacity must be < 2^30.  The device-side waits (grid barriers) are bounded; none can
 * hang.
 */
size_t gs_bin_sort_workspace_size(int64_t n, int64_t capacity, const gs_camera* cam);
gs_status gs_bin_sort(const float* proj, int64_t n, const gs_camera* cam, void* workspace,
                      size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                      uint32_t* ranges, int64_t* count, int64_t* count_host, void* stream);

/* ---------------------------------------------------------------------------
 * gs_bin_sort_batch -- gs_bin_sort for the `batch` views of one training step (the
 * Grendel-GS notes' batch of images, §4.2), with results identical to `batch` separate
 * gs_bin_sort calls.  The depth sorts of up to 8 views run in one launch, so their short,
 * barrier-bound phases overlap; the tile sorts follow view by view.
 *   projs      host array of `batch` device pointers, [3][n][4] each (one n for all views).
 *   cams       host array of `batch` cameras (image sizes may differ).
 *   workspace  gs_bin_sort_batch_workspace_size(batch, n, capacity, cams) bytes, 256-byte
 *              aligned: one set of capacity-sized tile-sort buffers plus depth-sort buffers
 *              for min(batch, 8) views.
 *   keys       host array of `batch` device pointers (entries may be NULL), or NULL.
 *   vals, ranges  host arrays of `batch` device pointers: view v's outputs, as gs_bin_sort's.
 *   counts     device int64 [batch][2]: view v's count[0], count[1] as gs_bin_sort's.
 *   counts_host optional host int64 [batch]: if non-NULL the call synchronises the stream,
 *              stores every M there and returns GS_ERR_CAPACITY / GS_ERR_TIMEOUT if any view
 *              reported it.
 * Argument checks are gs_bin_sort's, per view; batch must be >= 1.
 */
size_t gs_bin_sort_batch_workspace_size(int batch, int64_t n, int64_t capacity, const gs_camera* cams);
gs_status gs_bin_sort_batch(const float* const* projs, int batch, int64_t n, const gs_camera* cams,
                            void* workspace, size_t workspace_bytes, uint64_t* const* keys,
                            uint32_t* const* vals, int64_t capacity, uint32_t* const* ranges,
                            int64_t* counts, int64_t* counts_host, void* stream);

/* ---------------------------------------------------------------------------
 * gs_render_fwd -- per-pixel front-to-back alpha compositing of the tile's sorted list
 * (Grendel-GS notes, 训练流程 "图像渲染").  For pixel p and list entries j in order:
 *   d = p + 0.5 - (u, v); power = -(A dx^2 + C dy^2)/2 - B dx dy; skip if power > 0;
 *   alpha = min(0.99, opacity * exp(power)); skip if alpha < 1/255;
 *   T' = T (1 - alpha); stop before this entry if T' < 1e-4;
 *   C += colour * alpha * T; T = T'.
 *   image = C + T bg;  T_final = T;  n_contrib = 1 + list position of the last
 *   accumulated entry (0 if none).
 * bg is a host array of 3 floats (may be NULL for black).
 * work is optional (NULL: not written), [3][H][W] uint32: work[0] = list entries the pixel
 *   evaluated (through its termination point), work[1] = entries it accumulated, work[2] =
 *   entries its warp walked (the warp-culled list up to the point where all of the warp's
 *   pixels were done) -- the work counts behind the compositing kernels' roofline figures.
 * tile_order is optional (NULL: tiles in index order), [Tx*Ty] uint32, a permutation of the
 *   tile numbers (gs_tile_order): the order in which the tiles' thread blocks are issued.
 *   It changes no result, only how evenly the tiles' unequal work spreads over the SMs.
 * tile_cost is optional (NULL: not written), [Tx*Ty] uint32: per tile, the largest
 *   n_contrib of its pixels (the length of the backward's walk), for gs_tile_order.
 */
gs_status gs_render_fwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                        const gs_camera* cam, const float* bg, float* image, float* T_final,
                        uint32_t* n_contrib, uint32_t* work, const uint32_t* tile_order,
                        uint32_t* tile_cost, void* stream);

/* ---------------------------------------------------------------------------
 * gs_tile_order -- the order in which the compositing calls issue a view's tiles, heaviest
 * first.  Not a step of the method: a launch order for gs_render_fwd / gs_render_bwd (a
 * long tile issued last would run alone at the end of the launch).  A tile's cost is
 * tile_cost[t] if tile_cost is not NULL (gs_render_fwd's per-tile output, for the
 * backward), else its list length ranges[t][1] - ranges[t][0] (for the forward).  The
 * tiles_x x tiles_y grid is cut into square blocks of block x block tiles (block = 1..8;
 * smaller at the right and bottom edges); a block's key is that of its largest cost c: 0 for
 * c = 0, else
 * 1 + 16 floor(log2 c) + the four bits of c below its leading one (steps of 1/16 octave).
 * Writes order [tiles_x * tiles_y] uint32, a permutation of the tile numbers: blocks by
 * falling key, each block's tiles together in row-major order (neighbouring tiles run at
 * the same time and share Gaussians in L2); the order of blocks with equal keys is
 * unspecified.  One small launch; tiles_x, tiles_y <= 65535.
 */
gs_status gs_tile_order(const uint32_t* ranges, const uint32_t* tile_cost, int tiles_x, int tiles_y,
                        int block, uint32_t* order, void* stream);

/* ---------------------------------------------------------------------------
 * gs_loss -- L1 + SSIM image loss ("损失计算：L1 + SSIM 损失", Grendel-GS notes, 训练流程)
 * and its gradient.  Per view:
 *   loss = w_l1 * mean|I - I*| + w_ssim * (1 - mean SSIM),
 * means over all 3*H*W values; SSIM per channel with an 11x11 Gaussian window
 * (sigma 1.5, normalised), zero padding, C1 = 0.01^2, C2 = 0.03^2, sigma terms
 * E[x^2] - mu^2.  Writes dL_dimage = scale * dloss/dimage and
 *   *loss_dev = scale * loss          (accumulate == 0)
 *   *loss_dev += scale * loss         (accumulate != 0)
 * The loss value is reduced in a fixed order (deterministic).
 * workspace: gs_loss_workspace_size(width, height) bytes.
 */
size_t gs_loss_workspace_size(int width, int height);
gs_status gs_loss(const float* image, const float* target, int width, int height, float w_l1,
                  float w_ssim, float scale, float* loss_dev, int accumulate, float* dL_dimage,
                  void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * gs_loss_noalloc -- gs_loss without a workspace.  The paper has no counterpart for this
 * entry point: it is a calling convention of this library, not a step of the method.
 * For callers that cannot provide device memory: their memory is owned by another
 * allocator under a fixed budget, or they must not call cudaMalloc / cudaFree, which can
 * synchronise the whole device.  The partial sums live in a fixed array inside the
 * library's device image (512 KB, held by every GPU that loads the library until the
 * process exits), so the call allocates nothing.  Same arguments and results as gs_loss.
 *  - Limit: ceil(width/32) * ceil(height/32) * 3 <= 65536 (e.g. up to 4096 x 4096);
 *    larger images return GS_ERR_INVALID with the limit in the message.
 *  - Every call looks up the array's device address on the current device (a host-side
 *    runtime query that allocates nothing; not cached, so a device reset cannot leave a
 *    stale address).  The first call on a device also loads the library's device code
 *    there: make that first call before any stream capture.
 *  - Every call shares the one array: calls that overlap on the GPU (on different
 *    streams with no ordering between them) race and give wrong results.  Each call
 *    rewrites the parts it reads, so nothing needs clearing between calls.
 */
gs_status gs_loss_noalloc(const float* image, const float* target, int width, int height, float w_l1,
                          float w_ssim, float scale, float* loss_dev, int accumulate, float* dL_dimage,
                          void* stream);

/* ---------------------------------------------------------------------------
 * gs_render_bwd -- reverse-order backward of gs_render_fwd ("反向传播").  Walks each
 * pixel's list back to front from n_contrib, recovering T by T / (1 - alpha), and
 * writes per-Gaussian screen-space gradients into grad2d [n][12] (the call clears
 * grad2d first; contributions of all pixels are summed with atomics, so the
 * summation order, and the last bits, vary from run to run).  tile_order: as for
 * gs_render_fwd (NULL: index order); the backward's is best made from gs_render_fwd's
 * tile_cost.
 */
gs_status gs_render_bwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                        const gs_camera* cam, const float* bg, const float* T_final,
                        const uint32_t* n_contrib, const float* dL_dimage, float* grad2d,
                        const uint32_t* tile_order, void* stream);

/* ---------------------------------------------------------------------------
 * gs_project_bwd -- reverse mode of gs_project: grad2d -> parameter gradients,
 * ACCUMULATED (+=) into grads [15][n][4] so that a batch's views sum.  Only Gaussians
 * with radius > 0 in proj are touched.  Exact derivative of the forward, including the
 * quaternion normalisation, the clamped Jacobian, the view direction of the SH colour
 * and the colour clamp at 0.
 *   densify_stat  optional device float [n][2] (8-byte aligned), ACCUMULATED: for every
 *                 Gaussian with radius > 0 in this view, [0] += |(dL/du, dL/dv)| (the length of
 *                 its screen-space mean gradient, from grad2d) and [1] += 1 -- the statistic
 *                 gs_densify reads.  NULL: not accumulated.
 */
gs_status gs_project_bwd(const float* params, int64_t n, const gs_camera* cam, const float* proj,
                         const float* grad2d, float* grads, float* densify_stat, void* stream);

/* ---------------------------------------------------------------------------
 * gs_visible_sets -- per-view visible sets and their pairwise overlaps, the inputs of a
 * primitive-level RAW/WAW/WAR check (Odin summary §1 Jaccard weight w_ij = |Pi n Pj| /
 * |Pi u Pj|, 0 for an empty union; Odin article: the hook that collects the active
 * primitives after backward).
 *   proj_per_view  HOST array of `batch` device pointers to proj [3][n][4].
 *   V_b = {i : radius_b[i] > 0}.
 *   visible_bits  optional: the same sets as bitsets, [batch][bits_stride] uint32 (as
 *            gs_project_batch writes them); when given, the radius words are not read and
 *            proj_per_view may be NULL.  bits_stride >= ceil(n / 32).
 *   offsets  [batch + 1] int64; indices [batch * n] uint32: V_b ascending at
 *            indices[offsets[b] .. offsets[b+1]).
 *   union_idx [n] uint32 ascending; *n_union (device int64) = |U|, U = union of V_b.
 *   inter    [batch][batch] int64 = |V_i n V_j|.
 *   jaccard  [batch][batch] float = fp32 rounding of the exact ratio inter / |V_i u V_j|
 *            (computed in double from the integer counts), 0 when the union is empty.
 * workspace: gs_visible_sets_workspace_size(batch, n) bytes.  batch in [1, 64].  After the
 *   call the workspace begins with the views' bitsets, [batch][ceil(n / 32)] uint32 (bit
 *   i % 32 of word i / 32 of view b set iff i is in V_b), valid until the workspace is used
 *   again (gs_project_bwd_adam can take them).
 */
size_t gs_visible_sets_workspace_size(int batch, int64_t n);
gs_status gs_visible_sets(const float* const* proj_per_view, int batch, int64_t n, void* workspace,
                          size_t workspace_bytes, int64_t* offsets, uint32_t* indices,
                          uint32_t* union_idx, int64_t* n_union, int64_t* inter, float* jaccard,
                          const uint32_t* visible_bits, int64_t bits_stride, void* stream);

/* ---------------------------------------------------------------------------
 * gs_sparse_adam -- Adam on the listed Gaussians only, with the batch scaling rule of
 * the Grendel-GS notes §4.2: lr' = lr sqrt(batch), beta1' = beta1^batch,
 * beta2' = beta2^batch.  For every float of the listed Gaussians' 15 planes:
 *   m = beta1' m + (1 - beta1') g;  v = beta2' v + (1 - beta2') g^2;
 *   p -= lr' (m / (1 - beta1'^step)) / (sqrt(v / (1 - beta2'^step)) + eps);  g = 0
 * (the two bias corrections are applied as host-computed factors and the quotient by a
 * fast division: the update is exact to a few ulp).
 * Gaussians not listed keep p, m, v and g bit-for-bit.
 *   idx     union_idx from gs_visible_sets (strictly ascending, each < n).
 *   n_idx   DEVICE int64 count of idx entries (<= max_idx); read by the kernel so the
 *           call needs no host synchronisation.
 *   step    t >= 1, the number of batches applied so far including this one.
 *   counts  optional DEVICE array of n_counts int64[2] records from gs_bin_sort (one per
 *           view of the batch); if any record's status word (element [1]) is nonzero the
 *           whole update is skipped, so a batch whose binning overflowed leaves the
 *           parameters and moments untouched and can be re-run.  NULL: never skipped.
 */
gs_status gs_sparse_adam(float* params, float* grads, float* exp_avg, float* exp_avg_sq, int64_t n,
                         const uint32_t* idx, const int64_t* n_idx, int64_t max_idx, float lr,
                         float beta1, float beta2, float eps, int batch, int64_t step,
                         const int64_t* counts, int n_counts, void* stream);

/* ---------------------------------------------------------------------------
 * gs_project_bwd_adam -- the batch's backward projection and its update in one pass:
 * gs_project_bwd for every view b (gradients summed in view order, starting from zero)
 * followed by gs_sparse_adam over the Gaussians with radius > 0 in at least one view (the
 * union of the visible sets), except that the gradient planes are never written.
 * The pages have no counterpart for this entry point as a separate call: it is the
 * composition of the two steps above, fused so that the gradients stay on chip.
 *   cams, proj_per_view, grad2d_per_view  HOST arrays of `batch` entries (the latter two
 *              hold device pointers); batch in [1, 16].
 *   exp_avg, exp_avg_sq  Adam moments [15][n][4]; lr, beta1, beta2, eps, step as for
 *              gs_sparse_adam (batch scaling rule included); counts/n_counts likewise
 *              (any nonzero status word skips the whole update).
 *   densify_stat  optional, as for gs_project_bwd, summed over the batch's views (in view
 *              order); not touched when the update is skipped.
 *   visible_bits  optional (NULL: each view's radius words are read from its proj): the
 *              views' visible sets as bitsets, [batch][bits_stride] uint32, bit i % 32 of
 *              word i / 32 of view b set iff radius_b[i] > 0 -- what gs_visible_sets leaves
 *              at the start of its workspace.  bits_stride >= ceil(n / 32).  The results
 *              are the same; the bitsets replace 16 bytes of radius-word traffic per
 *              Gaussian and view with a bit.
 * Gaussians visible in no view keep p, m and v bit-for-bit.
 */
gs_status gs_project_bwd_adam(float* params, int64_t n, const gs_camera* cams, int batch,
                              const float* const* proj_per_view, const float* const* grad2d_per_view,
                              float* exp_avg, float* exp_avg_sq, float lr, float beta1, float beta2,
                              float eps, int64_t step, const int64_t* counts, int n_counts,
                              float* densify_stat, const uint32_t* visible_bits, int64_t bits_stride,
                              void* stream);

/* ---------------------------------------------------------------------------
 * gs_probe_ffma -- measurement utility with no counterpart in the method: `blocks` CTAs of
 * 256 threads each run `iters` iterations of eight independent fused multiply-adds and
 * write one float per thread to out[blocks * 256].  The caller times the launch:
 * blocks * 256 * iters * 16 flops over the elapsed time is the FP32 throughput the
 * compositing and loss fractions are reported against.
 */
gs_status gs_probe_ffma(float* out, int blocks, int iters, void* stream);

/* ---------------------------------------------------------------------------
 * Test hooks (no counterpart in the method).
 * gs_debug_set_wait_limit: iterations a device-side wait (a grid barrier of gs_bin_sort's
 *   cooperative launches) spins before it gives up and reports status bit 2 (default
 *   1 << 22; values < 1 restore it).
 * gs_debug_drop_publish: arms the next gs_bin_sort call only.  mode 1: CTA 0 of the tile
 *   sort never arrives at its first grid barrier; mode 2: the same in the depth sort; every
 *   other CTA's barrier wait then runs out; 0 disarms.  Used to test that the bounded waits
 *   report GS_ERR_TIMEOUT instead of hanging.
 */
void gs_debug_set_wait_limit(int64_t iterations);
void gs_debug_drop_publish(int mode);

/* ---------------------------------------------------------------------------
 * gs_tile_split -- pixel-wise load balancing of the Grendel-GS notes (§3.1: record each
 * 16x16 block's render time ET, CumSum = cumsum(ET), a target of Total / K per GPU, split
 * points by searchsorted).  The block "time" is an integer cost: the per-pixel costs in
 * cost_px (e.g. work[2] of gs_render_fwd, the entries each pixel's warp walked) summed over
 * the block, so the sums and the split points are exact.
 *   cost_px    [H][W] uint32 per-pixel costs.
 *   tile_cost  output, Tx * Ty uint64: each block's cost (row-major tiles).
 *   cum        output, Tx * Ty uint64: inclusive cumulative sum of tile_cost.
 *   bounds     output, parts + 1 int64: part k holds tiles [bounds[k], bounds[k + 1]);
 *              bounds[k] = number of tiles with parts * cum[i] <= k * Total (searchsorted on
 *              the right: a tile ending exactly on a target stays in the earlier part; a zero
 *              total puts every tile in part 0).
 * parts in 1..1024; 64-bit arrays 8-byte aligned.  Two kernels; no workspace.
 */
gs_status gs_tile_split(const uint32_t* cost_px, int width, int height, int parts, uint64_t* tile_cost,
                        uint64_t* cum, int64_t* bounds, void* stream);

/* ---------------------------------------------------------------------------
 * gs_view_order -- greedy schedule of a batch's views by the Odin summary's scheduling score
 * s(v | U_prev) = sum of w_uv over the previous set, with w the Jaccard weights of the
 * relative locality graph (gs_visible_sets' jaccard output).  The static schedule places
 * weakly coupled transitions next to each other: views are taken one at a time into task
 * units of `unit` views, the next being the unscheduled view with the smallest score against
 * the previous unit (ties: the lower index; the first unit's scores are 0).  Scores are
 * float32 sums over the previous unit in its scheduling order.
 *   weights  [batch][batch] float32.
 *   order    output, batch int32: the views in schedule order.
 *   score    output, batch float32: each scheduled view's score when it was taken.
 * batch in 1..64, unit in 1..batch.
 */
gs_status gs_view_order(const float* weights, int batch, int unit, int32_t* order, float* score, void* stream);

/* ---------------------------------------------------------------------------
 * gs_prune -- the pruning half of densification (Grendel-GS notes, 训练流程: "prune
 * low-opacity Gaussians").  Gaussian i is kept when its opacity logit (plane 0, w of the
 * first set) is >= min_logit, i.e. opacity >= sigmoid(min_logit) (a NaN logit is dropped),
 * and its 15 planes of every set move to the next free slot, index order preserved.
 *   planes_in   host array of n_sets (1..4) device pointers, [15][n][4] each; set 0 is the
 *               parameters (its logit decides), the others e.g. the Adam moments.
 *   planes_out  host array of n_sets device pointers, [15][out_stride][4] each, not
 *               overlapping the inputs; may be NULL when out_stride == 0 (count only).
 *   workspace   gs_prune_workspace_size(n) bytes, 256-byte aligned.
 *   n_keep      device int64[1]: the number kept (the true count even above out_stride;
 *               slots at or beyond out_stride are not written).
 *   n_keep_host optional host int64: if non-NULL the call synchronises, stores the count and
 *               returns GS_ERR_CAPACITY if it exceeds a nonzero out_stride.
 * A usual pass: once with out_stride = 0 to learn the count, then with out_stride = count.
 */
size_t gs_prune_workspace_size(int64_t n);
gs_status gs_prune(const float* const* planes_in, int n_sets, int64_t n, float min_logit,
                   float* const* planes_out, int64_t out_stride, void* workspace, size_t workspace_bytes,
                   int64_t* n_keep, int64_t* n_keep_host, void* stream);

/* ---------------------------------------------------------------------------
 * gs_densify -- the clone / split half of densification (Grendel-GS notes, 训练流程:
 * "致密化", clone or split the Gaussians that need more detail).  The pages give no
 * criterion; this library's reading, in its own terms:
 *   selected   densify_stat[i][1] > 0 and densify_stat[i][0] / densify_stat[i][1] >=
 *              grad_threshold (fp32): the mean, over the views that saw Gaussian i since the
 *              statistic was last cleared, of its screen-space mean-gradient length;
 *   split      a selected Gaussian whose largest log-scale is > log_scale_threshold; the
 *              others are cloned.
 * Output, [15][out_stride][4] planes of parameters and both Adam moments: the Gaussians not
 * split, in index order, moments kept; then, for every selected Gaussian in index order, its
 * new ones with zero moments: a clone (exact copy of the parameters), or two split children
 * k = 0, 1 with mean mu + R(q / |q|) (exp(log-scale) * z_k), z_k = normals[i][3k .. 3k + 2],
 * and log-scales lowered by ln 1.6, the other parameters copied.
 *   params, exp_avg, exp_avg_sq  [15][n][4], 16-byte aligned.
 *   densify_stat  [n][2] float (see gs_project_bwd); normals  [n][6] float, the caller's
 *              standard normal draws (two 3-vectors per Gaussian; only split ones are read).
 *   *_out      [15][out_stride][4], not overlapping the inputs; NULL with out_stride == 0
 *              (count only).  Slots at or beyond out_stride are not written.
 *   workspace  gs_densify_workspace_size(n) bytes, 256-byte aligned.
 *   counts     device int64[3]: output count, clones, splits (the true counts even above
 *              out_stride).  counts_host: optional host int64[3]; if non-NULL the call
 *              synchronises, stores them and returns GS_ERR_CAPACITY if the output count
 *              exceeds a nonzero out_stride.
 * A usual pass: once with out_stride = 0 to learn the count, then with out_stride = count.
 */
size_t gs_densify_workspace_size(int64_t n);
gs_status gs_densify(const float* params, const float* exp_avg, const float* exp_avg_sq, int64_t n,
                     const float* densify_stat, float grad_threshold, float log_scale_threshold,
                     const float* normals, float* params_out, float* exp_avg_out, float* exp_avg_sq_out,
                     int64_t out_stride, void* workspace, size_t workspace_bytes, int64_t* counts,
                     int64_t* counts_host, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GS_H_ */
