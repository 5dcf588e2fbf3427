"""Host threads calling the library at once (ctypes releases the GIL for
the duration of each call, so the calls really overlap in C): the fitter
gives every thread the program a lone call gives, and the program registry
never hands out a torn mix of two programs being installed concurrently."""
import threading

from polynomial_activation_gb300 import binding as B

ROWS = [(B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16, 4), (B.POLY_TANH, B.POLY_FWD, B.POLY_F16, 5),
        (B.POLY_SILU, B.POLY_BWD, B.POLY_BF16, 3), (B.POLY_GELU, B.POLY_FWD, B.POLY_F16, 6)]


def _run(workers):
    errors = []

    def wrap(f):
        def body():
            try:
                f()
            except BaseException as e:          # surfaced in the main thread
                errors.append(e)
        return body

    threads = [threading.Thread(target=wrap(f)) for f in workers]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
        assert not t.is_alive()
    if errors:
        raise errors[0]


def test_concurrent_fits_match_lone_fits():
    alone = {r: bytes(B.poly_fit(*r)) for r in ROWS}
    got = {r: [] for r in ROWS}
    _run([(lambda r=r: got[r].append(bytes(B.poly_fit(*r)))) for r in ROWS for _ in range(2)])
    for r in ROWS:
        assert got[r] == [alone[r], alone[r]], r


def test_registry_reads_are_never_torn():
    key = (B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16)
    p3, p5 = B.poly_fit(*key, 3), B.poly_fit(*key, 5)
    valid = {bytes(p3), bytes(p5)}
    stop = threading.Event()
    seen = set()

    def writer(p):
        def body():
            for _ in range(20000):
                B.poly_set_program(p)
        return body

    torn = []

    def reader():
        while not stop.is_set():
            q = bytes(B.poly_get_program(*key))
            if q not in valid:
                torn.append(q)
            seen.add(q)

    try:
        B.poly_set_program(p3)
        r = threading.Thread(target=reader)
        r.start()
        _run([writer(p3), writer(p5)])
        stop.set()
        r.join(timeout=60)
        assert not r.is_alive()
        assert not torn, f"{len(torn)} torn reads"
        assert seen and seen <= valid
        assert bytes(B.poly_get_program(*key)) in valid
    finally:
        stop.set()
        B.poly_reset_programs()
