"""The thin-input kernel's staging and tap arithmetic, modelled on the CPU (no GPU).

tc_gather.cu stages, per CTA and pass, one contiguous run of NHWC input rows in shared
memory and reads each output pixel's three taps of a row as the aligned 32-bit words that
cover them (a 0- or 16-bit funnel shift).  This model repeats that arithmetic -- the CTA's
pixel share, the pass bounds, the staged byte range, the word window -- for sampled pixels
of many shapes, and checks that (1) every word read lies between the weight tile that
precedes the staging buffer and the slack that follows it, and (2) each in-range tap read
from the modelled staging buffer is the input element the convolution needs.  The
constants are the kernel's: staging buffer, slack, the smallest weight tile, CTAs per SM.
"""
import random

import pytest

CAP = 32768     # staging buffer bytes
SLACK = 64      # bytes after it that tap reads may touch
B_MIN = 1024    # smallest weight tile in front of the staging buffer
R = S = 3


def ctas_per_sm(c):
    return 3 if c == 3 else 2


def cta_share(m, b, g):
    base, extra = m // g, m % g
    p0 = b * base + min(b, extra)
    return p0, p0 + base + (1 if b < extra else 0)


def pass_end(ps, p_end, wo, k):
    return min((ps // wo + k) * wo, p_end)


def pass_rows(p0, p1, howo, wo, h, sh, ph):
    ia, ib = p0 // howo, (p1 - 1) // howo
    oha, ohb = (p0 - ia * howo) // wo, (p1 - 1 - ib * howo) // wo
    lo, hi = oha * sh - ph, ohb * sh - ph + R - 1
    return ia * h + max(lo, 0), ib * h + min(hi, h - 1)


def pass_bytes(first, last, rb):
    gs = first * rb
    ge = (last + 1) * rb if last >= first else gs
    return gs, ge, gs & ~15


def choose_pass_rows(m, grid, h, ho, wo, sh, ph, rb):
    def fits(k):
        for b in range(grid):
            p0, p1 = cta_share(m, b, grid)
            ps = p0
            while ps < p1:
                pe = pass_end(ps, p1, wo, k)
                gs, ge, a0 = pass_bytes(*pass_rows(ps, pe, ho * wo, wo, h, sh, ph), rb)
                if ge - a0 > CAP:
                    return False
                ps = pe
        return True
    k = min((m + grid - 1) // grid // wo + 2, 1 << 20)
    k = max(1, min(k, (CAP // rb - R) // sh + 1))
    while k >= 1 and not fits(k):
        k -= 1
    return k


def check_shape(n, h, w, c, sh, sw, ph, pw, sms=152, rng=None):
    rng = rng or random.Random(0)
    ho, wo = (h + 2 * ph - R) // sh + 1, (w + 2 * pw - S) // sw + 1
    m = n * ho * wo
    rb = w * c * 2
    grid = min((m + 127) // 128, ctas_per_sm(c) * sms)
    k = choose_pass_rows(m, grid, h, ho, wo, sh, ph, rb)
    assert k >= 1
    nw = (6 * c + 5) // 4
    checked = 0
    for b in sorted(set([0, grid - 1] + rng.sample(range(grid), min(grid, 6)))):
        p0, p1 = cta_share(m, b, grid)
        ps = p0
        while ps < p1:
            pe = pass_end(ps, p1, wo, k)
            first, last = pass_rows(ps, pe, ho * wo, wo, h, sh, ph)
            gs, ge, a0 = pass_bytes(first, last, rb)
            xs = gs - a0  # staged row `first` starts here, from the staging buffer's start

            def byte(off):  # modelled staging buffer: element e of x holds e & 0xffff
                g = off - xs + gs
                if not (gs <= g < ge):
                    return 0xAB
                v = (g // 2) & 0xffff
                return v >> 8 if g & 1 else v & 0xff
            for p in rng.sample(range(ps, pe), min(pe - ps, 40)):
                img, rem = divmod(p, ho * wo)
                oh, ow = divmod(rem, wo)
                iw0 = ow * sw - pw
                for r in range(R):
                    ih = oh * sh - ph + r
                    rin = 0 <= ih < h
                    start = xs + (img * h - first + ih) * rb + iw0 * c * 2 if rin else xs
                    wa, shift = start & ~3, (start & 2) * 8
                    assert wa >= -B_MIN and wa + 4 * nw <= CAP + SLACK, (p, r, wa)
                    if not rin:
                        continue
                    words = [sum(byte(wa + 4 * j + q) << (8 * q) for q in range(4)) for j in range(nw)]
                    for kk in range(3 * c):
                        s_, ch = divmod(kk, c)
                        if not 0 <= iw0 + s_ < w:
                            continue
                        j, j1 = kk // 2, min(kk // 2 + 1, nw - 1)
                        two = ((words[j1] << 32 | words[j]) >> shift) & 0xffffffff
                        val = two >> 16 if kk & 1 else two & 0xffff
                        assert val == (((img * h + ih) * w + iw0 + s_) * c + ch) & 0xffff, (p, r, kk)
                        checked += 1
            ps = pe
    return checked


SHAPES = [
    (1, 640, 640, 3, 2, 2, 1, 1),   # the stem
    (8, 640, 640, 3, 2, 2, 1, 1),   # a batch of stems
    (1, 12, 1800, 3, 1, 1, 1, 1),   # the widest 3-channel rows that fit
    (2, 33, 35, 1, 1, 1, 1, 1),
    (3, 17, 19, 4, 2, 2, 1, 1),
    (2, 21, 23, 3, 1, 1, 0, 0),
    (1, 40, 41, 4, 1, 1, 2, 2),
    (2, 9, 7, 1, 2, 2, 0, 0),       # 14-byte rows
    (5, 6, 6, 4, 1, 1, 2, 2),       # pad 2, passes across images
    (2, 50, 50, 3, 3, 3, 0, 0),     # stride 3
]


@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_tap_words_in_bounds_and_exact(shape):
    assert check_shape(*shape, rng=random.Random(hash(shape) & 0xffff)) > 0


def test_padding_beyond_filter_minus_one_would_drop_a_row():
    """Why the kernel takes at most filter - 1 padding: with 4 rows of padding on a 3-row
    filter, a pass that ends in an image whose first output rows read only padding gets a
    last staged row from that image, below the previous image's last row."""
    h, ph = 27, 4
    ho, wo = (h + 2 * ph - R) + 1, 50
    howo = ho * wo
    # a pass from output row 30 of image 0 to output row 0 of image 1
    first, last = pass_rows(30 * wo, howo + 1, howo, wo, h, 1, ph)
    assert last < h - 1   # image 0's row 26, read by output row 30, is not staged
