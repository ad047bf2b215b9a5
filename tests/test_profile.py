"""The calibration profile's key check, on the CPU: a profile is accepted
only by the device and library that wrote it.  A matching profile passes;
one written for another GPU name, SM count, clock, compute capability or
library version is stale; a file that is not a profile (malformed, truncated,
wrongly formatted, nested without bound, missing) is an argument error."""
import json

import pytest

from dsmem_thread_block_gb300 import _credit as C


def _key(**kw):
    k = C.DeviceKey(gpu_name=b"NVIDIA GB300", sms=152, sm_clock_mhz=2070, mem_clock_mhz=3996,
                    cc_major=10, cc_minor=3)
    for f, v in kw.items():
        setattr(k, f, v)
    return k


def _profile(**over):
    d = {"format": "credit-profile-1", "library": C.credit_version(),
         "device": {"name": "NVIDIA GB300", "sms": 152, "sm_clock_mhz": 2070,
                    "mem_clock_mhz": 3996, "cc_major": 10, "cc_minor": 3},
         "dsmem": {"barrier_ns": [0.0] * 17, "exchange_ns": [0.0] * 17,
                   "async_exchange_ns": [0.0] * 17},
         "plans": []}
    for k, v in over.items():
        if k in d["device"]:
            d["device"][k] = v
        else:
            d[k] = v
    return d


@pytest.fixture(scope="module")
def lib():
    return C.load()


def _write(tmp_path, obj, name="p.json"):
    p = tmp_path / name
    p.write_text(obj if isinstance(obj, str) else json.dumps(obj))
    return str(p)


def test_matching_profile_is_accepted(lib, tmp_path):
    assert C.credit_profile_check(_write(tmp_path, _profile()), _key()) == C.OK


@pytest.mark.parametrize("field,value", [("gpu_name", b"NVIDIA B200"), ("sms", 148),
                                         ("sm_clock_mhz", 1965), ("mem_clock_mhz", 4000),
                                         ("cc_major", 9), ("cc_minor", 0)])
def test_profile_of_another_device_is_stale(lib, tmp_path, field, value):
    path = _write(tmp_path, _profile())
    assert C.credit_profile_check(path, _key(**{field: value})) == C.ERR_NOT_CALIBRATED


def test_profile_of_another_library_version_is_stale(lib, tmp_path):
    path = _write(tmp_path, _profile(library="0.0.1"))
    assert C.credit_profile_check(path, _key()) == C.ERR_NOT_CALIBRATED


@pytest.mark.parametrize("text", [
    "", "{", "[]", '{"format": "credit-profile-1"',
    json.dumps(_profile(format="something-else")),
    json.dumps({"library": "0.5.0"}),
    "[" * 1000 + "]" * 1000,
    '{"format": "credit-profile-1", "library": 5, "device": {}}',
    json.dumps(_profile()) + " trailing",
])
def test_malformed_profiles_are_rejected(lib, tmp_path, text):
    assert C.credit_profile_check(_write(tmp_path, text), _key()) == C.ERR_INVALID_ARG


def test_missing_profile_is_rejected(lib, tmp_path):
    assert C.credit_profile_check(str(tmp_path / "none.json"), _key()) == C.ERR_INVALID_ARG
