"""The barrier protocols of the attention kernels, run as executable models on the CPU
(tests/barrier_models.py).  The models cover the persistent dK/dV and dQ kernels, with random
item lists that include empty items and several CTAs on one counter, and the forward.  Random
interleavings of the warp roles, the copies and the MMAs must end, pass every parity wait at its
intended phase and never overwrite data before its readers are done.  Each model must also
catch every wait that is taken out of it."""
import pytest

from tests.barrier_models import DkdvModel, DkdvModel64, DqModel, PoolModel, run_forward_trials, run_trials

TRIALS = 150


@pytest.mark.parametrize("model", [DkdvModel, DkdvModel64, DqModel, PoolModel], ids=["dkdv", "dkdv64", "dq", "pool"])
def test_protocol_holds_on_random_schedules(model):
    err = run_trials(model, TRIALS)
    assert err is None, err


@pytest.mark.parametrize("model,wait", [
    (DkdvModel, "kvfree"), (DkdvModel, "empty"), (DkdvModel, "sfree"), (DkdvModel, "pfree"), (DkdvModel, "drain"),
    (DkdvModel64, "sfree"), (DkdvModel64, "pfree"), (DkdvModel64, "empty"),
    (DqModel, "qfree"), (DqModel, "kempty"), (DqModel, "vempty"), (DqModel, "sfree"), (DqModel, "pfree"),
    (DqModel, "dq"), (DqModel, "qt"),
    (PoolModel, "empty"), (PoolModel, "accfree"),
])
def test_model_catches_a_missing_wait(model, wait):
    # (the pooling's item_free wait is not in the list: with 8 item slots against a 2-deep stage
    # ring and two accumulators the producer never gets far enough ahead for it to bind; the
    # kernel keeps it all the same)
    assert run_trials(model, TRIALS, drop={wait}) is not None, f"{model.__name__} without {wait} passed"


def test_forward_protocol_holds_on_random_schedules():
    err = run_forward_trials(TRIALS)
    assert err is None, err


@pytest.mark.parametrize("wait", ["kempty", "vempty", "s_over_p", "odone"])
def test_forward_model_catches_a_missing_wait(wait):
    assert run_forward_trials(TRIALS, drop={wait}) is not None, f"forward without {wait} passed"


@pytest.mark.parametrize("model", [DkdvModel, DkdvModel64, DqModel, PoolModel], ids=["dkdv", "dkdv64", "dq", "pool"])
def test_abort_path_leaves_nothing_in_flight(model):
    """Waits expire at random: every role leaves its loops, and when the CTA frees its tensor
    memory and exits no copy or MMA is still in flight (and no drain waits forever)."""
    err = run_trials(model, 2 * TRIALS, expire=True)
    assert err is None, err


def test_forward_abort_path_leaves_nothing_in_flight():
    err = run_forward_trials(2 * TRIALS, expire=True)
    assert err is None, err


@pytest.mark.parametrize("model", [DkdvModel, DkdvModel64, DqModel, PoolModel, "fwd"], ids=["dkdv", "dkdv64", "dq", "pool", "fwd"])
@pytest.mark.parametrize("skipped", ["abort_drain", "abort_mma_drain"])
def test_model_catches_a_drain_skipped_on_abort(model, skipped):
    """Without the producer's drain of its issued copies, or with the issuers' drains giving
    up once the abort flag is up, some CTA exits with work in flight."""
    if model == "fwd":
        err = run_forward_trials(2 * TRIALS, drop={skipped}, expire=True)
    else:
        err = run_trials(model, 2 * TRIALS, drop={skipped}, expire=True)
    assert err is not None, f"{model} without {skipped} passed"
