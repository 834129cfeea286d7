"""Host-side pieces of bench.py that need no GPU: the guarded extra legs."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_leg_not_asked_for_is_not_run():
    b = _bench()
    errors = {}
    ran = []
    assert b.run_leg({"stress"}, "batched", lambda: ran.append(1), errors) is None
    assert ran == [] and errors == {}


def test_leg_result_is_returned():
    b = _bench()
    errors = {}
    assert b.run_leg({"batched"}, "batched", lambda: {"write_us": 1.5}, errors) == {"write_us": 1.5}
    assert errors == {}


def test_failing_leg_is_reported_not_raised():
    b = _bench()
    errors = {}

    def boom():
        raise RuntimeError("leg went wrong")

    assert b.run_leg({"stress", "batched"}, "stress", boom, errors) is None
    assert errors == {"stress": "RuntimeError: leg went wrong"}
    # the other legs still run
    assert b.run_leg({"stress", "batched"}, "batched", lambda: 3, errors) == 3
