"""Pins of the segment-parallel form (oracle/segment_scan.py): it equals the
token recurrence for any cut of the chunks into segments, including strong
decay, empty and partial sequences; and a segment's composed map is affine
in its entry state."""
import numpy as np
import pytest

import kda_inputs as KI
import oracle


def ref(d):
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"],
                            initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                            scale=d["scale"])


def scan(d, segments, chunk=16):
    return oracle.segment_scan(d["q"], d["k"], d["v"], d["g"], d["beta"],
                               initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"],
                               scale=d["scale"], segments=segments, chunk=chunk)


def close(a, b):
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12 * max(1.0, np.abs(b).max()))


@pytest.mark.parametrize("segments", [1, 2, 3, 7, 1000])
def test_segment_scan_equals_token_recurrence(segments):
    d = KI.make_case([100, 0, 37, 260], H=2, seed=41, init_state=True)
    o_r, f_r = ref(d)
    o, f = scan(d, segments)
    close(o, o_r)
    close(f, f_r)


def test_segment_scan_strong_decay_odd_chunk():
    d = KI.make_case([123], H=1, seed=42, init_state=False)
    d["g"][:, :, ::3] = -8.0
    o_r, f_r = ref(d)
    o, f = scan(d, 4, chunk=7)
    close(o, o_r)
    close(f, f_r)


def test_segment_map_is_affine_in_the_entry_state():
    """Two runs that differ only in the initial state end with final states
    whose difference is the same linear map (the composed M) applied to the
    initial difference: here checked through linearity, f(2 S) - f(S) =
    f(S) - f(0)."""
    d = KI.make_case([90], H=1, seed=43, init_state=True)
    s = d["initial_state"].double()
    out = []
    for factor in (0.0, 1.0, 2.0):
        e = dict(d, initial_state=s * factor)
        out.append(scan(e, 3)[1])
    close(out[2] - out[1], out[1] - out[0])
