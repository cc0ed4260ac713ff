"""CPU-side checks of the C-ABI library (no GPU needed): it loads, exports every
symbol include/motion.h declares, validates arguments on the host, and its host
helpers follow the score / PSNR definitions.  Also the source contracts of the
kernels and the separation between the product and the oracle."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "motion.h")
CSRC = os.path.join(ROOT, "integer_image_filter_gb300", "csrc")


@pytest.fixture(scope="module")
def lib():
    import integer_image_filter_gb300 as iif
    from integer_image_filter_gb300 import _build
    _build.build()
    return iif.load_library()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^MOTION_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ("motion_init", "motion_submit", "motion_submit_batch", "psnr_sse",
                     "psnr_sse_yuv420_batch", "motion_psnr_yuv420_batch"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_names_match_the_header():
    import integer_image_filter_gb300 as iif
    for name in declared_functions():
        assert name in iif.EXPORTED_SYMBOLS
        if name != "motion_last_cuda_error":
            assert callable(getattr(iif, name))


def test_host_argument_validation(lib):
    import ctypes
    h = ctypes.c_void_p()
    assert lib.motion_init(2, 10, 8, ctypes.byref(h)) == 2          # too small
    assert lib.motion_init(10, 2, 8, ctypes.byref(h)) == 2
    assert lib.motion_init(10, 10, 7, ctypes.byref(h)) == 3         # bpc
    assert lib.motion_init(10, 10, 17, ctypes.byref(h)) == 3
    assert lib.motion_init(40000, 10, 8, ctypes.byref(h)) == 5      # too large
    assert lib.motion_init(10, 10, 8, None) == 1
    assert lib.psnr_sse(None, None, 16, 16, 8, 8, 7, None, None) == 3
    assert lib.psnr_sse(None, None, 16, 16, 0, 8, 8, None, None) == 1
    assert lib.motion_destroy(None) == 0
    assert lib.motion_reset(None) == 1
    assert lib.motion_submit_batch(None, None, 0, 0, 0, None, None) == 1


def test_layout_validation_before_any_device_call(lib):
    """Context-free batch calls check every plane layout on the host and
    return before touching the device: pitches shorter than a row, odd
    16-bit layouts, and frame spans that leave a 48-bit address space.  Every
    case here must fail validation: the pointers are not device memory."""
    import ctypes
    p = ctypes.c_void_p(4096)                     # never dereferenced: validation fails first
    out = ctypes.cast(ctypes.c_void_p(4096), ctypes.POINTER(ctypes.c_uint64))
    W, H = 64, 32

    def yuv(n, py, puv, sy, suv, bpc=8):
        return lib.psnr_sse_yuv420_batch(W, H, bpc, n, p, p, p, p, p, p, py, puv, sy, suv, None, out)

    def moments(n, pitch, stride, bpc=8):
        return lib.moment_sums_batch(W, H, bpc, n, p, p, pitch, stride, None, out)

    assert yuv(2, W - 1, W // 2, W * H, W * H // 4) == 4          # luma pitch < row
    assert yuv(2, W, W // 2 - 1, W * H, W * H // 4) == 4          # chroma pitch < row
    assert yuv(2, 2 * W + 1, W, 2 * W * H, W * H // 2, bpc=10) == 4   # odd 16-bit pitch
    assert yuv(2, W, W // 2, 1 << 47, W * H // 4) == 1            # stride beyond 2^46
    assert yuv(1 << 10, W, W // 2, 1 << 40, W * H // 4) == 1      # 2^50 bytes of frames
    assert moments(2, W - 1, W * H) == 4
    assert moments(3, W, 1 << 47) == 1
    assert moments(1 << 12, W, 1 << 37) == 1                     # 2^49 bytes
    assert moments(1 << 20, W, (1 << 28) + 16) == 1               # just over 2^48
    assert moments(2, W, W * H, bpc=17) == 3
    assert moments(-1, W, W * H) == 1


def test_noalloc_layout_validation_before_any_device_call(lib):
    """The allocation-free entry point applies the same layout checks as the
    context calls (pitch <= 2^40, stride <= 2^46, n frames within 2^48
    bytes, 16-bit alignment) and refuses before any CUDA call: a frame stride
    above 2^63 would otherwise turn negative as a signed offset."""
    import ctypes
    p = ctypes.c_void_p(4096)                     # never dereferenced: validation fails first
    out = ctypes.cast(ctypes.c_void_p(4096), ctypes.POINTER(ctypes.c_uint64))
    W, H = 64, 32

    def call(n, pitch, stride, bpc=8, frames=p, cont=0):
        return lib.motion_submit_batch_noalloc(frames, n, W, H, bpc, stride, pitch, cont, None, out)

    assert call(2, W - 1, W * H) == 4                       # pitch < row
    assert call(2, 2 * W + 1, 2 * W * H, bpc=10) == 4       # odd 16-bit pitch
    assert call(2, 2 * W, 2 * W * H + 1, bpc=10) == 4       # odd 16-bit stride
    assert call(2, (1 << 40) + 16, W * H) == 1              # pitch beyond 2^40
    assert call(2, W, 1 << 47) == 1                         # stride beyond 2^46
    assert call(2, W, (1 << 63) + 16) == 1                  # stride above 2^63
    assert call(1 << 12, W, 1 << 37) == 1                   # 2^49 bytes of frames
    assert call(2, W, W * H, frames=None) == 1
    assert call(2, W, W * H, bpc=7) == 3
    assert lib.motion_submit_batch_noalloc(p, 2, 2, H, 8, W * H, W, 0, None, out) == 2
    assert lib.motion_submit_batch_noalloc(p, 1, 4096, 4096, 8, 0, 4096, 0, None, out) == 5
    assert lib.motion_noalloc_device_error(None, None) == 1


def test_init_without_device_reports_it(lib):
    import ctypes
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    h = ctypes.c_void_p()
    assert lib.motion_init(64, 48, 8, ctypes.byref(h)) == 8


def test_strerror_names_every_status(lib):
    import integer_image_filter_gb300 as iif
    for code in range(11):
        assert iif.motion_strerror(code) != "unknown status"
    assert iif.motion_strerror(99) == "unknown status"


def test_scores_helper_matches_definition(lib, oracle):
    import integer_image_filter_gb300 as iif
    rng = np.random.default_rng(5)
    sad = rng.integers(0, 2**40, size=33).astype(np.uint64)
    sad[0] = 0
    for (w, h) in ((64, 48), (3840, 2160), (3, 3)):
        s, m2 = iif.motion_scores_from_sad(sad, w, h)
        so, m2o = oracle.scores(sad, w, h)
        assert np.array_equal(s, so) and np.array_equal(m2, m2o)
        s, m2 = iif.motion_scores_from_sad(sad, w, h, next_score=0.5)
        so, m2o = oracle.scores(sad, w, h, next_score=0.5)
        assert np.array_equal(m2, m2o)
    assert iif.motion_scores_from_sad(np.zeros(0, np.uint64), 4, 4)[0].size == 0


def test_psnr_helper(lib):
    import oracle
    import integer_image_filter_gb300 as iif
    mse, db = iif.psnr_from_sse(0, 100, 8)
    assert mse == 0.0 and db == float("inf")
    for sse, n, bpc in ((100, 100, 8), (12345, 999, 10), (7, 3, 16)):
        mse, db = iif.psnr_from_sse(sse, n, bpc)
        assert mse == sse / n
        assert abs(db - oracle.psnr_db(sse, n, bpc)) <= 1e-12 * abs(db)


def test_binding_refuses_short_buffers(lib):
    """The binding checks every buffer it can measure before the library sees a
    pointer: outputs must be contiguous 64-bit arrays of the right length and
    inputs must reach their last sample (raised on the host, no GPU needed)."""
    import torch

    import integer_image_filter_gb300 as iif
    f = torch.zeros((2, 8, 8), dtype=torch.uint8)
    short = "are needed"
    with pytest.raises(ValueError, match=short):             # out: 4 of 8 values
        iif.moment_sums_batch(f, f, 8, torch.zeros((1, 4), dtype=torch.int64))
    with pytest.raises(TypeError, match="64-bit"):           # 32-bit output
        iif.moment_sums_batch(f, f, 8, torch.zeros((2, 4), dtype=torch.int32))
    with pytest.raises(ValueError, match="contiguous"):      # non-contiguous output
        iif.moment_sums_batch(f, f, 8, torch.zeros((4, 4), dtype=torch.int64)[::2])
    with pytest.raises(ValueError, match=short):             # pitch runs past the frames
        iif.moment_sums_batch(f, f, 8, torch.zeros((2, 4), dtype=torch.int64), pitch=16,
                              stride=64)
    with pytest.raises(ValueError, match=short):
        iif.motion_submit_batch_noalloc(f, torch.zeros(1, dtype=torch.int64))
    y, c = torch.zeros((3, 8, 8), dtype=torch.uint8), torch.zeros((3, 4, 4), dtype=torch.uint8)
    c2 = torch.zeros((2, 4, 4), dtype=torch.uint8)           # chroma of 2 pairs only
    with pytest.raises(ValueError, match=short):
        iif.psnr_sse_yuv420_batch(8, 8, 8, y, c, c2, y, c, c, torch.zeros((3, 3), dtype=torch.int64))
    with pytest.raises(ValueError, match=short):
        iif.motion_psnr_yuv420_batch_host(0, y.numpy(), c.numpy(), c.numpy(), y.numpy(),
                                          c.numpy(), c.numpy(), np.zeros(2, np.uint64))
    with pytest.raises(ValueError, match=short):             # host frames: 2 of 3 SADs
        iif.motion_submit_batch_host(0, y.numpy(), np.zeros(2, np.uint64))
    with pytest.raises(TypeError, match="64-bit"):
        iif.motion_submit_batch_host(0, y.numpy(), np.zeros(3, np.uint32))


def test_frame_chunk_plan(lib):
    """Launch sizing by SM count: the chunk counts that forced-chunk timings
    on a GB300 (608 resident CTAs, the block order of motion_tile_order) found
    fastest, and the invariants of the plan (1..8 chunks, at least 5 frames per
    chunk, one chunk for one frame)."""
    import integer_image_filter_gb300 as iif
    plan = iif.motion_plan_chunks
    assert plan(3840, 2160, 50, 608) == 2      # fused 4K 4:2:0 pairs (+2 % over one and three)
    assert plan(3840, 2160, 32, 608) == 1      # 10-bit 4K, batch 32 (+1 % over two, +4 % over three)
    assert plan(3840, 2160, 16, 608) == 1      # (+3.5 % over two)
    assert plan(1920, 1080, 32, 608) == 3      # (+4 % over two, +1.5 % over four, +6 % over one)
    assert plan(1920, 1080, 16, 608) in (1, 3)  # a tie, +2 % over two
    assert plan(1920, 1080, 8, 608) == 1
    assert plan(576, 324, 48, 608) == 8        # 55 tiles: as many chunks as allowed
    for (w, h) in ((64, 48), (576, 324), (1920, 1080), (3840, 2160), (8192, 4320)):
        for n in (0, 1, 2, 5, 9, 10, 31, 64, 300):
            for slots in (1, 152, 608, 1216):
                c = plan(w, h, n, slots)
                assert 1 <= c <= 8
                assert c == 1 or -(-n // c) >= 5, (w, h, n, slots, c)
                if n <= 1:
                    assert c == 1
    with pytest.raises(iif.MotionError):
        plan(0, 10, 4, 608)
    with pytest.raises(iif.MotionError):
        plan(10, 10, 4, 0)


def test_launch_blocks_cover_every_frame_once(lib):
    """The blocks of a batched launch (uniform chunks or a split tail) cover
    every (tile, frame) exactly once; a split tail keeps the tiles of the full
    waves whole, gives the last-wave tiles short chunks (at least 4 frames) and
    puts them after the whole tiles."""
    import numpy as np

    import integer_image_filter_gb300 as iif
    cases = [(3840, 2160, 32, 608, 32), (3840, 2160, 16, 608, 32), (3840, 2160, 50, 608, 32),
             (1920, 1080, 16, 608, 32), (1920, 1080, 32, 608, 32), (576, 324, 48, 608, 32),
             (64, 48, 4, 608, 32), (3840, 2160, 120, 608, 32), (4096, 2048, 9, 100, 32),
             (1000, 700, 13, 7, 32), (3, 3, 1, 1, 32), (1366, 768, 8, 152, 32),
             # 128 x 16 tiles (1064 resident on GB300): 1080p x 16 in one wave, a split
             # tail past one wave, ragged last tile rows
             (1920, 1080, 16, 1064, 16), (576, 324, 48, 1064, 16), (1920, 1080, 32, 900, 16),
             (1000, 700, 13, 7, 16), (3, 3, 1, 1, 16), (130, 17, 5, 1064, 16)]
    for (w, h, n, slots, rows) in cases:
        gx, gy = -(-w // 128), -(-h // rows)
        count, _ = iif.motion_launch_blocks(w, h, n, slots, tile_rows=rows)
        seen = np.zeros((gy, gx, n), np.int32)
        lens = []
        for b in range(count):
            _, (tx, ty, f0, f1) = iif.motion_launch_blocks(w, h, n, slots, b, tile_rows=rows)
            assert 0 <= tx < gx and 0 <= ty < gy and 0 <= f0 < f1 <= n, (w, h, n, b)
            seen[ty, tx, f0:f1] += 1
            lens.append(f1 - f0)
        assert (seen == 1).all(), (w, h, n, slots)
        tiles = gx * gy
        if rows == 32:
            c = iif.motion_plan_chunks(w, h, n, slots)
            assert (count != tiles * -(-n // -(-n // c))) == (count > tiles and lens[0] == n)
        if count > tiles and lens[0] == n:
            # a split tail: whole tiles first, then chunks of >= 4 frames
            rest = tiles % slots
            whole = tiles - rest
            assert all(x == n for x in lens[:whole]), (w, h, n)
            chunk = max(lens[whole:])
            assert 4 <= chunk < n, (w, h, n)
            # every chunk has that length but the one that ends at the last frame
            for b in range(whole, count):
                _, (tx, ty, f0, f1) = iif.motion_launch_blocks(w, h, n, slots, b, tile_rows=rows)
                assert f1 - f0 == chunk or f1 == n, (w, h, n, b)
            assert 0 < 2 * rest <= slots
    # the 10-bit 4K batch of 32: 1824 whole tiles and 216 tiles in two halves
    assert iif.motion_launch_blocks(3840, 2160, 32, 608)[0] == 1824 + 2 * 216
    assert iif.motion_launch_blocks(3840, 2160, 32, 608, 1824)[1][2:] == (0, 16)
    assert iif.motion_launch_blocks(3840, 2160, 32, 608, 1824 + 216)[1][2:] == (16, 32)
    with pytest.raises(iif.MotionError):
        iif.motion_launch_blocks(3840, 2160, 32, 608, 1824 + 432)
    # the fused 4:2:0 launch of 50 pairs takes the split tail ahead of two uniform
    # chunks (the uniform plan alone would pick two)
    assert iif.motion_plan_chunks(3840, 2160, 50, 608) == 2
    assert iif.motion_launch_blocks(3840, 2160, 50, 608)[0] == 1824 + 2 * 216
    assert iif.motion_launch_blocks(3840, 2160, 50, 608, 1823)[1][2:] == (0, 50)
    assert iif.motion_launch_blocks(3840, 2160, 50, 608, 1824)[1][2:] == (0, 25)
    assert iif.motion_launch_blocks(3840, 2160, 50, 608, 1824 + 216)[1][2:] == (25, 50)
    with pytest.raises(iif.MotionError):
        iif.motion_launch_blocks(1920, 1080, 16, 608, tile_rows=24)
    # 1080p x 16 in 128 x 16 tiles: 1020 blocks of all 16 frames, one wave of 1064; the
    # last block takes the last interior tile (rows 1..66 interior, 67 on the border)
    assert iif.motion_launch_blocks(1920, 1080, 16, 1064, tile_rows=16)[0] == 1020
    assert iif.motion_launch_blocks(1920, 1080, 16, 1064, 1019, tile_rows=16)[1] == (14, 66, 0, 16)


def test_launch_shape(lib):
    """Motion-only launches whose 128 x 32 tiles, in their planned chunks, fit in
    one wave (608 resident blocks on GB300) take 128 x 16 tiles; the others,
    motion_v2's two-chunk 1080p plan among them, keep 128 x 32."""
    import integer_image_filter_gb300 as iif
    shape = iif.motion_launch_shape
    assert shape(1920, 1080, 16, 608) == 16           # 510 tiles, one chunk
    assert shape(1920, 1080, 32, 608) == 32           # three chunks: 1530 blocks
    assert shape(1920, 1080, 16, 608, v2=True) == 32  # motion_v2 plans two chunks
    assert shape(3840, 2160, 32, 608) == 32           # 2040 tiles
    assert shape(576, 324, 48, 608) == 16             # 55 tiles x 8 chunks = 440
    assert shape(64, 48, 1, 608) == 16
    assert shape(1920, 1080, 16, 500) == 32           # 510 tiles > 500
    for (w, h, n) in ((1920, 1080, 16), (3840, 2160, 32), (576, 324, 48), (3, 3, 1)):
        tiles = -(-w // 128) * -(-h // 32)
        c = iif.motion_plan_chunks(w, h, n, 608)
        assert (shape(w, h, n, 608) == 16) == (tiles * c <= 608)
    for bad in ((0, 10, 1, 608), (10, 10, 0, 608), (10, 10, 1, 0), (40000, 10, 1, 608)):
        with pytest.raises(iif.MotionError):
            shape(*bad)


def test_tile_order(lib):
    """Block order of a batched launch: every (tile, chunk) exactly once; the
    tiles that run the border copy of the frame loop (top row, rows whose halo
    passes the bottom edge, a partial last column) first; then the full tiles
    whose staged rows all lie in the frame -- left and right edge columns
    included -- in row-major order within each chunk."""
    import integer_image_filter_gb300 as iif
    order = iif.motion_tile_order
    for (w, h, chunks) in ((3840, 2160, 2), (1920, 1080, 3), (576, 324, 8), (64, 48, 1),
                           (129, 33, 2), (130, 34, 1), (258, 66, 3), (390, 98, 4), (1, 1, 1),
                           (32768, 40, 2), (40, 32768, 1), (8192, 4320, 1)):
        gx, gy = -(-w // 128), -(-h // 32)
        seen = set()
        kinds, interior = [], []
        for b in range(gx * gy * chunks):
            tx, ty, cz = order(w, h, chunks, b)
            assert 0 <= tx < gx and 0 <= ty < gy and 0 <= cz < chunks
            seen.add((tx, ty, cz))
            x0, y0 = 128 * tx, 32 * ty
            kinds.append(x0 + 128 <= w and y0 > 0 and y0 + 34 <= h)
            if kinds[-1]:
                interior.append((cz, ty, tx))
        assert len(seen) == gx * gy * chunks, (w, h, chunks)
        n_border = len(kinds) - sum(kinds)
        assert not any(kinds[:n_border]) and all(kinds[n_border:]), (w, h, chunks)
        assert interior == sorted(interior), (w, h, chunks)      # row-major per chunk
    for bad in ((0, 10, 1, 0), (10, 10, 0, 0), (10, 10, 9, 0), (10, 10, 1, 1), (10, 10, 1, -1),
                (32769, 10, 1, 0)):
        with pytest.raises(iif.MotionError):
            order(*bad)


# ---------------------------------------------------------------- source contracts
def _kernel_sources():
    return {f: open(os.path.join(CSRC, f)).read() for f in os.listdir(CSRC)
            if f.endswith((".cu", ".cuh"))}


# a single thread, warp 0 whose lanes each own one (frame, accumulator), or
# the last warp of the block to finish a window of frames, whose lanes each
# own one frame
_GUARD = re.compile(r"if \((lane|tid|threadIdx\.x|warp) == \d|if \(__shfl_sync\(0xffffffffu, last, 0\)\)")
_SHARED = re.compile(r"__shared__[^;]*?\b(\w+)\[")


def _single_lane_guarded(src: str, pos: int) -> bool:
    """True when the statement at pos, or one of the blocks enclosing it, is
    under an `if (lane|tid|threadIdx.x == k ...)` condition."""
    line_start = src.rfind("\n", 0, pos) + 1
    if _GUARD.search(src[line_start:pos]):
        return True
    prev_start = src.rfind("\n", 0, max(line_start - 1, 0)) + 1
    prev = src[prev_start:line_start].strip()
    if _GUARD.search(prev) and not prev.endswith((";", "{", "}")):
        return True          # `if (...)` on the line before, without braces
    depth = 0
    i = pos
    while i > 0:
        i -= 1
        c = src[i]
        if c == "}":
            depth += 1
        elif c == "{":
            if depth == 0:
                header_start = src.rfind("\n", 0, i) + 1
                if _GUARD.search(src[header_start:i]):
                    return True
            else:
                depth -= 1
    return False


def contract_violations(src: str) -> list:
    """Checks in the spirit of a kernel source contract: no cluster multicast,
    every atomic on an output is a 64-bit add issued once per block per
    accumulator (inside a lane-guarded branch; adds into the block's own
    shared-memory sums are exempt), no runtime index into kernel-parameter
    arrays."""
    bad = []
    if "multicast::cluster" in src:
        bad.append("cluster multicast")
    shared = set(_SHARED.findall(src))
    for m in re.finditer(r"\batomicAdd\(([^;]*)\);", src):
        target = re.match(r"\s*&(\w+)\[", m.group(1))
        if target and target.group(1) in shared:
            continue         # a block-local sum in shared memory, not an output
        if not _single_lane_guarded(src, m.start()):
            line_start = src.rfind("\n", 0, m.start()) + 1
            bad.append("atomic not guarded by a single lane: " + src[line_start:m.end()].strip())
    if re.search(r"\ba\.\w+\[[^\]]*(threadIdx|blockIdx|plane|lane)", src):
        bad.append("runtime index into a kernel-parameter array")
    return bad


def test_kernel_source_contract():
    for name, src in _kernel_sources().items():
        assert contract_violations(src) == [], name
    tile = _kernel_sources()["motion_tile.cu"]
    # the vertical pass writes a V tile that the horizontal pass reads
    assert "sV" in tile and "vtap(" in tile


@pytest.mark.parametrize("plant", [
    'asm("op.multicast::cluster");',
    "    atomicAdd(a.sad_out + f, t0);",
    "    __shared__ unsigned wsum[4];\n    atomicAdd(&out[f], t0);",
    "    const uint8_t* p = a.planes[plane];",
])
def test_contract_catches_planted_regressions(plant):
    assert contract_violations(plant + "\n") != []


def test_product_and_oracle_are_separate():
    pkg = os.path.join(ROOT, "integer_image_filter_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
                assert "oracle.c" not in text and "liboracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "integer_image_filter_gb300" not in text and "motion.h" not in text, f
