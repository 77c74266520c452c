"""B300-native (sm_103a) LaCT fast-weight chunk step: liblact.so + its binding."""
from . import lact  # noqa: F401
